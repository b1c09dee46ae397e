"""ctypes binding of libbf16_linear.so — argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into (pointer, size, stream) arguments, checks dtype /
contiguity / device on the Python side (the dtype guards the vLLM PR #42562
review asked for: both x and W must be bfloat16), and raises on a nonzero
status.  There is no fallback: if the library is missing the import-time
loader raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbf16_linear.so")

OK, EINVAL, EALIGN, EARCH, ELAUNCH, ETIMEOUT, EUNSUPPORTED, ENOSCRATCH = 0, -1, -2, -3, -4, -5, -6, -7
FLAG_PDL = 1      # weights read before the grid-dependency wait
FLAG_SERIAL = 2   # no programmatic dependent launch
(KERNEL_DOTPROD, KERNEL_SPLITK, KERNEL_TILE, KERNEL_SPLITK_WS, KERNEL_STREAM, KERNEL_TILE2, KERNEL_WARPROW,
 KERNEL_WARPMMA, KERNEL_DOTMMA, KERNEL_DOTMMA_WS, KERNEL_TILE_T) = range(11)
KERNEL_NAMES = {KERNEL_DOTPROD: "dotprod", KERNEL_SPLITK: "splitk", KERNEL_TILE: "tile",
                KERNEL_SPLITK_WS: "splitk_ws", KERNEL_STREAM: "stream", KERNEL_TILE2: "tile2",
                KERNEL_WARPROW: "warprow", KERNEL_WARPMMA: "warpmma", KERNEL_DOTMMA: "dotmma",
                KERNEL_DOTMMA_WS: "dotmma_ws", KERNEL_TILE_T: "tile_t"}


class Plan(ctypes.Structure):
    """Mirror of bf16l_plan in include/bf16_linear.h."""
    _fields_ = [("kernel", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("rows_per_cta", ctypes.c_int32), ("tokens_per_cta", ctypes.c_int32),
                ("split_k", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("flags", ctypes.c_int32), ("chunks_per_stage", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {f[0]: int(getattr(self, f[0])) for f in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(d["kernel"], "?")
        return d

    def __repr__(self):
        return f"Plan({self.as_dict()})"


class Device(ctypes.Structure):
    """Mirror of bf16l_device."""
    _fields_ = [("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32), ("num_sms", ctypes.c_int32)]


class Call(ctypes.Structure):
    """Mirror of bf16l_call (the argument block of bf16_linear_run)."""
    _fields_ = [("x", ctypes.c_void_p), ("W", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32), ("out_f32", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("plan", ctypes.POINTER(Plan)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("stream", ctypes.c_void_p)]


class BF16LinearError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is missing: build it with `python -m moe_router_gemm_gb300.build` "
                              "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.bf16_linear.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        lib.bf16_linear.restype = i32
        lib.bf16_linear_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.c_uint32, vp]
        lib.bf16_linear_ex.restype = i32
        lib.bf16_linear_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, ctypes.c_size_t, ctypes.c_uint32, vp]
        lib.bf16_linear_host.restype = i32
        lib.bf16_linear_host_staging_bytes.argtypes = [i32, i32, i32, i32]
        lib.bf16_linear_host_staging_bytes.restype = ctypes.c_size_t
        lib.bf16_linear_f32out.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.c_uint32, vp]
        lib.bf16_linear_f32out.restype = i32
        lib.bf16_linear_f32out_with_plan.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(Plan), vp]
        lib.bf16_linear_f32out_with_plan.restype = i32
        lib.bf16_linear_with_plan.argtypes = [vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(Plan), vp]
        lib.bf16_linear_with_plan.restype = i32
        lib.bf16_linear_plan.argtypes = [i32, i32, i32, ctypes.POINTER(Plan)]
        lib.bf16_linear_plan.restype = i32
        lib.bf16_linear_plan_for_device.argtypes = [i32, i32, i32, ctypes.POINTER(Device), ctypes.POINTER(Plan)]
        lib.bf16_linear_plan_for_device.restype = i32
        lib.bf16_linear_plan_check.argtypes = [i32, i32, i32, ctypes.POINTER(Device), ctypes.POINTER(Plan)]
        lib.bf16_linear_plan_check.restype = i32
        lib.bf16_linear_run.argtypes = [ctypes.POINTER(Call)]
        lib.bf16_linear_run.restype = i32
        lib.bf16_linear_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(Plan)]
        lib.bf16_linear_workspace_size.restype = ctypes.c_size_t
        lib.bf16_linear_plan_ws.argtypes = [i32, i32, i32, ctypes.POINTER(Device), ctypes.c_size_t,
                                            ctypes.POINTER(Plan)]
        lib.bf16_linear_plan_ws.restype = i32
        lib.bf16_linear_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
        lib.bf16_linear_noalloc.restype = i32
        lib.bf16_quant_fp8.argtypes = [vp, vp, vp, ctypes.c_int64, ctypes.c_uint32, vp]
        lib.bf16_quant_fp8.restype = i32
        lib.bf16_linear_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_uint32, vp]
        lib.bf16_linear_fp8.restype = i32
        lib.bf16_linear_fp8_with_plan.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(Plan), vp]
        lib.bf16_linear_fp8_with_plan.restype = i32
        lib.bf16_linear_fp8_split.argtypes = [i32, i32, i32, i32]
        lib.bf16_linear_fp8_split.restype = i32
        lib.bf16_quant_mxfp8.argtypes = [vp, ctypes.c_int64, i32, vp, vp, ctypes.c_uint32, vp]
        lib.bf16_quant_mxfp8.restype = i32
        lib.bf16_linear_mxfp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_uint32, vp]
        lib.bf16_linear_mxfp8.restype = i32
        lib.bf16_linear_mxfp8_with_plan.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.POINTER(Plan), vp]
        lib.bf16_linear_mxfp8_with_plan.restype = i32
        lib.bf16_linear_mxfp8_split.argtypes = [i32, i32, i32, i32, i32]
        lib.bf16_linear_mxfp8_split.restype = i32
        lib.bf16_linear_probe_read.argtypes = [vp, ctypes.c_size_t, i32, i32, vp, ctypes.c_uint32, vp]
        lib.bf16_linear_probe_read.restype = i32
        lib.bf16_linear_noalloc_scratch_bytes.argtypes = []
        lib.bf16_linear_noalloc_scratch_bytes.restype = ctypes.c_size_t
        lib.bf16_linear_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), i32]
        lib.bf16_linear_device_status.restype = i32
        lib.bf16_linear_selftest_wait.argtypes = [ctypes.c_uint32, vp]
        lib.bf16_linear_selftest_wait.restype = i32
        lib.bf16_linear_strerror.argtypes = [i32]
        lib.bf16_linear_strerror.restype = ctypes.c_char_p
        lib.bf16_linear_cuda_error.argtypes = []
        lib.bf16_linear_cuda_error.restype = i32
        lib.bf16_linear_version.argtypes = []
        lib.bf16_linear_version.restype = i32
        _lib = lib
        return lib


def strerror(status: int) -> str:
    return load().bf16_linear_strerror(int(status)).decode()


def _raise(status: int, what: str):
    lib = load()
    extra = ""
    if status == ELAUNCH:
        extra = f" (cuda error {lib.bf16_linear_cuda_error()})"
    raise BF16LinearError(status, f"{what}: {strerror(status)}{extra}")


def plan(M: int, N: int, K: int, device: tuple[int, int, int] | None = None) -> Plan:
    """The kernel and parameters chosen for (M, N, K); device = (cc_major, cc_minor, num_sms)."""
    p = Plan()
    if device is None:
        st = load().bf16_linear_plan(int(M), int(N), int(K), ctypes.byref(p))
    else:
        st = load().bf16_linear_plan_for_device(int(M), int(N), int(K), ctypes.byref(Device(*device)),
                                                ctypes.byref(p))
    if st != OK:
        _raise(st, f"bf16_linear_plan({M},{N},{K})")
    return p


def plan_check(M: int, N: int, K: int, p: Plan, device: tuple[int, int, int] | None = None) -> Plan:
    """Validate an explicit plan for (M, N, K); fills p.grid, raises BF16LinearError if unusable."""
    dev = Device(*device) if device is not None else None
    st = load().bf16_linear_plan_check(int(M), int(N), int(K), ctypes.byref(dev) if dev is not None else None,
                                       ctypes.byref(p))
    if st != OK:
        _raise(st, f"bf16_linear_plan_check({M},{N},{K}, {p})")
    return p


def plan_ws(M: int, N: int, K: int, workspace_bytes: int, device: tuple[int, int, int] | None = None) -> Plan:
    """The dispatcher's choice when `workspace_bytes` of workspace are available."""
    p = Plan()
    dev = Device(*device) if device is not None else None
    st = load().bf16_linear_plan_ws(int(M), int(N), int(K), ctypes.byref(dev) if dev is not None else None,
                                    int(workspace_bytes), ctypes.byref(p))
    if st != OK:
        _raise(st, f"bf16_linear_plan_ws({M},{N},{K})")
    return p


def workspace_size(M: int, N: int, K: int, p: Plan | None = None) -> int:
    """Workspace bytes a call needs (for plan p, else for the dispatcher's choice with workspace allowed)."""
    return int(load().bf16_linear_workspace_size(int(M), int(N), int(K), ctypes.byref(p) if p is not None else None))


def make_plan(kernel: int | str, **fields) -> Plan:
    """Build an explicit plan (for with_plan); unspecified fields are 0."""
    if isinstance(kernel, str):
        kernel = {v: k for k, v in KERNEL_NAMES.items()}[kernel]
    p = Plan()
    p.kernel = int(kernel)
    for k, v in fields.items():
        setattr(p, k, int(v))
    return p


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check(x, W, bias, out, out_dtype=None):
    import torch
    if x.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError(f"x and W must be torch.bfloat16 (got {x.dtype}, {W.dtype})")
    if bias is not None and bias.dtype != torch.bfloat16:
        raise TypeError(f"bias must be torch.bfloat16 (got {bias.dtype})")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError(f"need x[M,K] and W[N,K], got {tuple(x.shape)} and {tuple(W.shape)}")
    M, K = x.shape
    N = W.shape[0]
    if bias is not None and tuple(bias.shape) != (N,):
        raise ValueError(f"bias must be [{N}], got {tuple(bias.shape)}")
    for name, t in (("x", x), ("W", W), ("bias", bias)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    odt = out_dtype or torch.bfloat16
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=x.device)
    elif out.dtype != odt or tuple(out.shape) != (M, N) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError(f"out must be a contiguous CUDA {odt} tensor of shape [M, N]")
    devs = {t.device for t in (x, W, bias, out) if t is not None}
    if len(devs) != 1:
        raise ValueError(f"all tensors must be on one device, got {devs}")
    return M, N, K, out


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def host_staging_bytes(M: int, N: int, K: int, with_bias: bool) -> int:
    """Device staging bytes bf16_linear_host needs (bf16_linear_host_staging_bytes)."""
    return int(load().bf16_linear_host_staging_bytes(int(M), int(N), int(K), 1 if with_bias else 0))


def new_host_staging(M: int, N: int, K: int, with_bias: bool, device=None):
    """A device staging tensor for bf16_linear_host (the caching allocator aligns blocks to 512 bytes)."""
    import torch
    return torch.empty(max(256, host_staging_bytes(M, N, K, with_bias)), dtype=torch.uint8,
                       device=device or "cuda")


def bf16_linear_host(x, W, bias=None, out=None, *, staging, flags: int = 0, stream=None):
    """bf16_linear_host: x[M,K], W[N,K], bias[N] and out[M,N] are CPU bf16 tensors (page-locked for
    asynchronous copies; out is allocated page-locked when None); the library copies them through the
    CUDA tensor `staging`, runs the planned kernel and copies out back, all on the given (or current)
    stream.  Returns out, complete once the stream has reached the final copy."""
    import torch
    for name, t in (("x", x), ("W", W), ("bias", bias)):
        if t is not None and (t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CPU bf16 tensor")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError(f"need x[M,K] and W[N,K], got {tuple(x.shape)} and {tuple(W.shape)}")
    M, K = x.shape
    N = W.shape[0]
    if bias is not None and tuple(bias.shape) != (N,):
        raise ValueError(f"bias must be [{N}], got {tuple(bias.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    elif out.dtype != torch.bfloat16 or out.is_cuda or tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU bf16 tensor of shape [M, N]")
    if not staging.is_cuda or not staging.is_contiguous():
        raise ValueError("staging must be a contiguous CUDA tensor")
    dev = staging.device
    if torch.cuda.current_device() == dev.index:  # (entering a device context costs more than the call)
        h = _stream_handle(stream, dev)
        st = load().bf16_linear_host(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K, _ptr(staging),
                                     staging.numel() * staging.element_size(), int(flags), h)
    else:
        with torch.cuda.device(dev):
            st = load().bf16_linear_host(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K, _ptr(staging),
                                         staging.numel() * staging.element_size(), int(flags),
                                         _stream_handle(stream, dev))
    if st != OK:
        _raise(st, f"bf16_linear_host(M={M}, N={N}, K={K})")
    return out


def bf16_linear(x, W, bias=None, out=None, stream=None):
    """out[M,N] = x[M,K] @ W[N,K]^T (+ bias[N]) in bf16, on the given (or current) stream."""
    import torch
    M, N, K, out = _check(x, W, bias, out)
    with torch.cuda.device(x.device):
        st = load().bf16_linear(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                                _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_linear(M={M}, N={N}, K={K})")
    return out


def run(x, W, bias=None, out=None, *, out_f32=False, flags=0, plan_: Plan | None = None, workspace=None,
        stream=None):
    """The general entry point (bf16_linear_run): optional explicit plan and workspace tensor."""
    import torch
    M, N, K, out = _check(x, W, bias, out, out_dtype=torch.float32 if out_f32 else torch.bfloat16)
    c = Call()
    c.x, c.W, c.bias, c.out = x.data_ptr(), W.data_ptr(), (bias.data_ptr() if bias is not None else None), \
        out.data_ptr()
    c.M, c.N, c.K = M, N, K
    c.out_f32 = 1 if out_f32 else 0
    c.flags = int(flags)
    c.plan = ctypes.pointer(plan_) if plan_ is not None else None
    if workspace is not None:
        if not workspace.is_cuda or workspace.device != x.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor on the inputs' device")
        c.workspace = workspace.data_ptr()
        c.workspace_bytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(x.device):
        c.stream = _stream_handle(stream, x.device).value
        st = load().bf16_linear_run(ctypes.byref(c))
    if st != OK:
        _raise(st, f"bf16_linear_run(M={M}, N={N}, K={K}, plan={plan_})")
    return out


def bf16_linear_with_plan(x, W, bias=None, out=None, plan_: Plan | None = None, stream=None, workspace=None):
    """Run exactly `plan_` (no fallback: an unusable plan raises)."""
    if plan_ is None:
        raise ValueError("plan_ is required")
    return run(x, W, bias, out, plan_=plan_, workspace=workspace, stream=stream)


def new_workspace(nbytes: int, device=None):
    """A zero-filled workspace tensor of at least nbytes (256-byte aligned by the caching allocator)."""
    import torch
    return torch.zeros(max(256, int(nbytes)), dtype=torch.uint8, device=device or "cuda")


def bf16_linear_f32out(x, W, bias=None, out=None, stream=None, flags: int = 0, plan_: Plan | None = None):
    """fp32 out[M,N] = x @ W^T (+ bias): the router-logits variant (no rounding to bf16)."""
    import torch
    M, N, K, out = _check(x, W, bias, out, out_dtype=torch.float32)
    with torch.cuda.device(x.device):
        if plan_ is None:
            st = load().bf16_linear_f32out(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K, int(flags),
                                           _stream_handle(stream, x.device))
        else:
            st = load().bf16_linear_f32out_with_plan(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                                                     ctypes.byref(plan_), _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_linear_f32out(M={M}, N={N}, K={K})")
    return out


def bf16_linear_ex(x, W, bias=None, out=None, flags: int = 0, stream=None):
    """bf16_linear with BF16L_FLAG_* launch flags (1 = programmatic dependent launch)."""
    import torch
    M, N, K, out = _check(x, W, bias, out)
    with torch.cuda.device(x.device):
        st = load().bf16_linear_ex(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K, int(flags),
                                   _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_linear_ex(M={M}, N={N}, K={K})")
    return out


def bf16_linear_noalloc(x, W, bias=None, out=None, stream=None):
    """bf16 out = x @ W^T (+ bias) for callers that cannot allocate device memory.

    Runs the workspace split-K kernel with its scratch in the library's fixed
    device array (see bf16_linear.h); the library allocates nothing.  Pass
    `out` to avoid the allocation this wrapper would otherwise make for it.
    Calls share the array: keep them on one stream.
    """
    import torch
    M, N, K, out = _check(x, W, bias, out)
    with torch.cuda.device(x.device):
        st = load().bf16_linear_noalloc(_ptr(x), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                                        _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_linear_noalloc(M={M}, N={N}, K={K})")
    return out


def quant_fp8(x, scale, out=None, flags: int = 0, stream=None):
    """Static per-tensor quantisation (bf16_quant_fp8): bf16 x -> e4m3 codes (torch.uint8, same shape).

    `scale` is a one-element fp32 CUDA tensor (read on the device)."""
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError(f"x must be torch.bfloat16 (got {x.dtype})")
    if scale.dtype != torch.float32 or scale.numel() != 1 or not scale.is_cuda:
        raise ValueError("scale must be a one-element float32 CUDA tensor")
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    elif out.dtype != torch.uint8 or out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 tensor shaped like x")
    with torch.cuda.device(x.device):
        st = load().bf16_quant_fp8(_ptr(x), _ptr(scale), _ptr(out), x.numel(), int(flags),
                                   _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_quant_fp8(n={x.numel()})")
    return out


def bf16_linear_fp8(xq, wq, scale_x, scale_w, bias=None, out=None, flags: int = 0, stream=None,
                    plan_: Plan | None = None):
    """Per-tensor FP8 linear (bf16_linear_fp8): e4m3 codes xq[M,K], wq[N,K] (torch.uint8),
    one-element fp32 CUDA scale tensors, optional bf16 bias[N]; bf16 out[M,N]."""
    import torch
    for name, t in (("xq", xq), ("wq", wq)):
        if t.dtype != torch.uint8 or t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D uint8 (e4m3 code) CUDA tensor")
    for name, t in (("scale_x", scale_x), ("scale_w", scale_w)):
        if t.dtype != torch.float32 or t.numel() != 1 or not t.is_cuda:
            raise ValueError(f"{name} must be a one-element float32 CUDA tensor")
    M, K = xq.shape
    N = wq.shape[0]
    if wq.shape[1] != K:
        raise ValueError(f"need xq[M,K] and wq[N,K], got {tuple(xq.shape)} and {tuple(wq.shape)}")
    if bias is not None and (bias.dtype != torch.bfloat16 or tuple(bias.shape) != (N,) or not bias.is_cuda):
        raise ValueError(f"bias must be a bf16 CUDA tensor of shape ({N},)")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=xq.device)
    with torch.cuda.device(xq.device):
        if plan_ is None:
            st = load().bf16_linear_fp8(_ptr(xq), _ptr(wq), _ptr(scale_x), _ptr(scale_w), _ptr(bias), _ptr(out),
                                        M, N, K, int(flags), _stream_handle(stream, xq.device))
        else:
            st = load().bf16_linear_fp8_with_plan(_ptr(xq), _ptr(wq), _ptr(scale_x), _ptr(scale_w), _ptr(bias),
                                                  _ptr(out), M, N, K, ctypes.byref(plan_),
                                                  _stream_handle(stream, xq.device))
    if st != OK:
        _raise(st, f"bf16_linear_fp8(M={M}, N={N}, K={K})")
    return out


def quant_mxfp8(x, out=None, scales=None, flags: int = 0, stream=None):
    """MXFP8 quantisation (bf16_quant_mxfp8) of a contiguous bf16 CUDA tensor x[rows, K], K % 32 == 0:
    returns (codes uint8 [rows, K], scales uint8 [rows, K / 32])."""
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D bf16 CUDA tensor")
    rows, K = x.shape
    if out is None:
        out = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((rows, max(1, K // 32)), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        st = load().bf16_quant_mxfp8(_ptr(x), rows, K, _ptr(out), _ptr(scales), int(flags),
                                     _stream_handle(stream, x.device))
    if st != OK:
        _raise(st, f"bf16_quant_mxfp8(rows={rows}, K={K})")
    return out, scales


def bf16_linear_mxfp8(xq, xs, wq, ws, bias=None, out=None, flags: int = 0, stream=None, plan_: Plan | None = None):
    """MXFP8 linear (bf16_linear_mxfp8): e4m3 codes xq[M,K], wq[N,K] (uint8) with E8M0 block scales
    xs[M,K/32], ws[N,K/32] (uint8), optional bf16 bias[N]; bf16 out[M,N]."""
    import torch
    for name, t in (("xq", xq), ("wq", wq), ("xs", xs), ("ws", ws)):
        if t.dtype != torch.uint8 or t.dim() != 2 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D uint8 CUDA tensor")
    M, K = xq.shape
    N = wq.shape[0]
    if wq.shape[1] != K or tuple(xs.shape) != (M, K // 32) or tuple(ws.shape) != (N, K // 32):
        raise ValueError(f"shapes xq{tuple(xq.shape)} xs{tuple(xs.shape)} wq{tuple(wq.shape)} ws{tuple(ws.shape)}")
    if bias is not None and (bias.dtype != torch.bfloat16 or tuple(bias.shape) != (N,) or not bias.is_cuda):
        raise ValueError(f"bias must be a bf16 CUDA tensor of shape ({N},)")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=xq.device)
    with torch.cuda.device(xq.device):
        h = _stream_handle(stream, xq.device)
        if plan_ is None:
            st = load().bf16_linear_mxfp8(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(bias), _ptr(out), M, N, K,
                                          int(flags), h)
        else:
            st = load().bf16_linear_mxfp8_with_plan(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), _ptr(bias), _ptr(out),
                                                    M, N, K, ctypes.byref(plan_), h)
    if st != OK:
        _raise(st, f"bf16_linear_mxfp8(M={M}, N={N}, K={K})")
    return out


def mxfp8_split(M: int, N: int, K: int, threads: int = 128, num_sms: int = 152) -> int:
    """The K split bf16_linear_mxfp8 uses (host logic, no GPU)."""
    return int(load().bf16_linear_mxfp8_split(M, N, K, threads, num_sms))


def fp8_split(M: int, N: int, K: int, num_sms: int = 152) -> int:
    """The K split bf16_linear_fp8 uses for a shape (host logic, no GPU)."""
    return int(load().bf16_linear_fp8_split(M, N, K, num_sms))


def probe_read(src, grid: int, threads: int, sink, nbytes: int | None = None, stream=None, flags: int = 0):
    """Launch the read-floor probe (bf16_linear_probe_read) over the bytes of the CUDA tensor `src`
    (the first nbytes of them, or none when src is None); CTA b XORs its checksum into sink[b] of the
    int32 CUDA tensor `sink` (at least `grid` elements).  flags: 0 (the library's launch mode) or
    FLAG_SERIAL."""
    import torch
    if sink is not None and sink.numel() < grid:
        raise ValueError(f"sink needs {grid} elements, has {sink.numel()}")
    nb = 0 if src is None else (src.numel() * src.element_size() if nbytes is None else int(nbytes))
    dev = sink.device if sink is not None else torch.device("cuda", torch.cuda.current_device())
    st = load().bf16_linear_probe_read(_ptr(src), nb, int(grid), int(threads), _ptr(sink), int(flags),
                                       _stream_handle(stream, dev))
    if st != OK:
        _raise(st, f"bf16_linear_probe_read(bytes={nb}, grid={grid}, threads={threads})")


def device_status(clear: bool = False) -> int:
    """The device's kernel status word (0 = no kernel wait gave up).  Synchronises."""
    v = ctypes.c_int32(0)
    st = load().bf16_linear_device_status(ctypes.byref(v), int(bool(clear)))
    if st != OK:
        _raise(st, "bf16_linear_device_status")
    return int(v.value)


def selftest_wait(limit_us: int, stream=None):
    """Launch the bounded-wait diagnostic (see bf16_linear.h)."""
    import torch
    st = load().bf16_linear_selftest_wait(int(limit_us), _stream_handle(stream, torch.cuda.current_device()))
    if st != OK:
        _raise(st, "bf16_linear_selftest_wait")


def version() -> int:
    return int(load().bf16_linear_version())
