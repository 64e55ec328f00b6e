"""GB300-native MoE decode routing: router GEMV, top-k gate, sort, MXFP8 quant.

Thin Python binding over the C ABI of libmoe_route.so (include/moe_route.h):
the functions below have the ABI's names without the ``mr_`` prefix, check
dtypes/devices/contiguity, allocate outputs with torch when none are given,
and pass raw pointers plus torch's current CUDA stream.  Every step of the
path runs in the library's CUDA kernels; there is no other implementation
behind these calls.  If the library is missing or fails to load, every call
raises.

bf16 tensors are torch.bfloat16; MXFP8 codes and E8M0 scales are uint8.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "MoeRouteError", "MoeRouteUnsupported", "Scratch", "library_path", "load_library",
    "set_launch_flags", "get_launch_flags", "LAUNCH_PDL", "LAUNCH_TEST_STALL", "LAUNCH_LEGACY_MMA",
    "LAUNCH_TEST_SLOW_SIGMOID", "LAUNCH_CHECK_SCRATCH", "set_wait_limit_ns",
    "device_error", "router_gemv_supported", "scratch_bytes", "sort_capacity", "router_gemv", "route_topk",
    "moe_sort", "mxfp8_quant", "moe_route_sort_quant", "router_gemv_noalloc", "shared_gate_up", "moe_route",
    "PreparedRoute", "moe_sort_quant", "mxfp4_quant", "norm_apply", "moe_route_sort_quant_norm",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_route.so")
_lib = None

(MR_OK, MR_ERR_UNSUPPORTED, MR_ERR_INVALID_ARG, MR_ERR_SCRATCH_TOO_SMALL, MR_ERR_CUDA, MR_ERR_TIMEOUT,
 MR_ERR_SCRATCH_DIRTY) = range(7)
SCORING = {"softmax": 0, "sigmoid": 1}
NORM_KIND = {"rms": 0, "gemma": 1}
QUANT_FORMAT = {None: 0, "mxfp8": 1, "mxfp4": 2}
SCRATCH_COUNTER_BYTES = 32768
PSORT_MAX_ASSIGN = 65536   # mr_moe_sort: one launch, no scratch, up to this many assignments
QUANT_SORTED_ROWS = 0x100  # mr_moe_sort_quant: quantised rows in sorted order


class MoeRouteError(RuntimeError):
    """The library rejected the call or CUDA reported an error."""

    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {_load().mr_status_string(status).decode()}"
        if status == MR_ERR_CUDA:
            msg += f" (cudaError_t {_load().mr_last_cuda_error()})"
        super().__init__(msg)


class MoeRouteUnsupported(MoeRouteError):
    """The shape is outside what the kernels cover (MR_ERR_UNSUPPORTED)."""


def library_path() -> str:
    return _LIB_PATH


# (name, restype, argtypes) of every exported symbol; the ABI test checks this
# list against include/moe_route.h.
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "mr_status_string": (ctypes.c_char_p, [_I]),
    "mr_abi_version": (_I, []),
    "mr_set_launch_flags": (_I, [_I]),
    "mr_get_launch_flags": (_I, []),
    "mr_router_gemv_supported": (_I, [_I, _I, _I, _I64]),
    "mr_scratch_bytes": (_SZ, [_I, _I, _I, _I]),
    "mr_scratch_reset": (_I, [_P, _SZ, _P]),
    "mr_router_gemv": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "mr_route_topk": (_I, [_P, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "mr_sort_capacity": (_I64, [_I, _I, _I, _I]),
    "mr_moe_sort": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _I64, _P, _SZ, _P]),
    "mr_mxfp8_quant": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "mr_moe_route_sort_quant": (_I, [_P, _I64, _P, _I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P,
                                     _P, _P, _P, _I64, _P, _P, _P, _SZ, _P]),
    "mr_router_gemv_noalloc": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P]),
    "mr_moe_route_sort_quant_norm": (_I, [_P, _I64, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P,
                                          _P, _P, _P, _I64, _P, _P, _P, _SZ, _P]),
    "mr_norm_apply": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "mr_mxfp4_quant": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "mr_moe_route": (_I, [_P, _P]),
    "mr_moe_sort_quant": (_I, [_P, _I, _I, _I, _I, _P, _I64, _I, _I, _P, _P, _P, _I64, _P, _P, _P]),
    "mr_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "mr_device_error": (_I, [_I]),
    "mr_shared_gate_up": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P]),
    "mr_last_cuda_error": (_I, []),
}


def load_library(path: str | None = None):
    """Load libmoe_route.so (built by decode_expert_routing_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libmoe_route.so not found at {p}: build it with "
            "`python -m decode_expert_routing_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


_load = load_library


def _check(status: int, what: str):
    if status == MR_OK:
        return
    if status == MR_ERR_UNSUPPORTED:
        raise MoeRouteUnsupported(status, what)
    raise MoeRouteError(status, what)


# ---------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _stream_ptr(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_ptr(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _row_major_2d(x, name):
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with a contiguous last dimension")
    return x.stride(0)


def _one_device(**tensors):
    """The one CUDA device of every given tensor (None entries skipped)."""
    devs = {}
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        devs.setdefault(t.device, name)
    if len(devs) != 1:
        raise ValueError("tensors on different devices: " + ", ".join(f"{n} on {d}" for d, n in devs.items()))
    return next(iter(devs))


def _check_out(t, name, shape, dtype, device, min_numel=False):
    """A caller-passed output: contiguous, of this dtype and shape (or at
    least this many elements when min_numel), on this device."""
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if min_numel:
        if t.numel() < shape:
            raise ValueError(f"{name} needs at least {shape} elements, has {t.numel()}")
    elif tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _check_scratch(scratch, device):
    if scratch is not None and scratch.tensor.device != device:
        raise ValueError(f"scratch must be on {device}")


def _launch_ctx(device):
    """The calling thread's current device set to device for the C call (the
    library launches on the current device, on the given stream)."""
    return _torch().cuda.device(device)


def _stream_on(device, stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


LAUNCH_PDL = 1
LAUNCH_TEST_STALL = 2  # test hook: the cluster kernels' bounded waits run out
LAUNCH_LEGACY_MMA = 4  # router GEMV of more than 64 rows: split-K mma.sync kernel instead of tcgen05
LAUNCH_TEST_SLOW_SIGMOID = 8  # test hook: every exact sigmoid score through its double-double path
LAUNCH_CHECK_SCRATCH = 16  # debug: calls that use scratch counters verify they are zero first (synchronous)


def set_launch_flags(flags: int) -> None:
    """Process-wide launch options (LAUNCH_PDL: programmatic dependent launch)."""
    _check(_load().mr_set_launch_flags(int(flags)), "mr_set_launch_flags")


def get_launch_flags() -> int:
    return int(_load().mr_get_launch_flags())


def set_wait_limit_ns(ns: int) -> None:
    """Limit of every bounded wait inside the cluster kernels (default 1 s)."""
    _check(_load().mr_set_wait_limit_ns(int(ns)), "mr_set_wait_limit_ns")


def device_error(clear: bool = False) -> int:
    """MR_OK, or MR_ERR_TIMEOUT once a bounded wait ran out on the current
    device (synchronous; call after the streams have finished)."""
    st = int(_load().mr_device_error(int(clear)))
    if st not in (MR_OK, MR_ERR_TIMEOUT):
        _check(st, "mr_device_error")
    return st


def router_gemv_supported(M: int, N: int, K: int, ldx: int | None = None) -> bool:
    return bool(_load().mr_router_gemv_supported(M, N, K, K if ldx is None else ldx))


def scratch_bytes(M_max: int, N: int, K: int, topk: int) -> int:
    return int(_load().mr_scratch_bytes(M_max, N, K, topk))


def sort_capacity(M: int, topk: int, N: int, block: int) -> int:
    return int(_load().mr_sort_capacity(M, topk, N, block))


class Scratch:
    """A caller-owned scratch buffer (torch uint8 on a CUDA device), zeroed
    once at creation; every call of the library leaves it reusable."""

    def __init__(self, M_max: int, N: int, K: int, topk: int, device=None):
        torch = _torch()
        self.nbytes = scratch_bytes(M_max, N, K, topk)
        if self.nbytes == 0:
            raise ValueError("scratch size query rejected the arguments")
        self.tensor = torch.empty(self.nbytes, dtype=torch.uint8,
                                  device=device if device is not None else "cuda")
        self.reset()

    def reset(self, stream=None):
        _check(_load().mr_scratch_reset(ctypes.c_void_p(self.tensor.data_ptr()), self.nbytes,
                                        _stream_ptr(stream)), "mr_scratch_reset")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())

    def counters(self):
        """The counter prefix as int32 (all zero between calls)."""
        return self.tensor[:SCRATCH_COUNTER_BYTES].view(_torch().int32)


# ---------------------------------------------------------------- the path

def router_gemv(x, w, out=None, scratch: Scratch | None = None, stream=None):
    """fp32 logits [M, N] = x [M, K] (bf16) @ w [N, K]^T (bf16)."""
    torch = _torch()
    dev = _one_device(x=x, w=w, out=out)
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dim() != 2 or not w.is_contiguous() or w.shape[1] != K:
        raise ValueError("w must be contiguous [N, K]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    _check_out(out, "out", (M, N), torch.float32, dev)
    if scratch is None:
        scratch = Scratch(M, N, K, 1, device=dev)
    _check_scratch(scratch, dev)
    with _launch_ctx(dev):
        _check(_load().mr_router_gemv(_dev_ptr(x, "x", torch.bfloat16), ldx, _dev_ptr(w, "w", torch.bfloat16),
                                      _dev_ptr(out, "out", torch.float32), M, N, K, scratch.ptr,
                                      scratch.nbytes, _stream_on(dev, stream)), "mr_router_gemv")
    return out


def router_gemv_noalloc(x, w, out=None, stream=None):
    """Router GEMV using the library's own fixed-size device scratch (no
    scratch argument, nothing allocated by the library).  For callers that
    cannot allocate; calls on one device share that scratch, so overlapping
    calls race.  The first call per device does a one-time set-up."""
    torch = _torch()
    dev = _one_device(x=x, w=w, out=out)
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    N = w.shape[0]
    if w.dim() != 2 or not w.is_contiguous() or w.shape[1] != K:
        raise ValueError("w must be contiguous [N, K]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
    _check_out(out, "out", (M, N), torch.float32, dev)
    with _launch_ctx(dev):
        _check(_load().mr_router_gemv_noalloc(_dev_ptr(x, "x", torch.bfloat16), ldx,
                                              _dev_ptr(w, "w", torch.bfloat16),
                                              _dev_ptr(out, "out", torch.float32), M, N, K,
                                              _stream_on(dev, stream)), "mr_router_gemv_noalloc")
    return out


def route_topk(logits, topk: int, scoring: str = "softmax", bias=None, renormalize: bool = True,
               ids=None, weights=None, stream=None):
    """(topk_ids int32 [M, k], topk_weights fp32 [M, k])."""
    torch = _torch()
    dev = _one_device(logits=logits, bias=bias, ids=ids, weights=weights)
    if logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be contiguous [M, N]")
    M, N = logits.shape
    if bias is not None:
        _check_out(bias, "bias", (N,), torch.float32, dev)
    if ids is None:
        ids = torch.empty((M, topk), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((M, topk), dtype=torch.float32, device=dev)
    _check_out(ids, "ids", (M, topk), torch.int32, dev)
    _check_out(weights, "weights", (M, topk), torch.float32, dev)
    with _launch_ctx(dev):
        _check(_load().mr_route_topk(_dev_ptr(logits, "logits", torch.float32), M, N, topk, SCORING[scoring],
                                     _dev_ptr(bias, "bias", torch.float32, allow_none=True), int(renormalize),
                                     _dev_ptr(ids, "ids", torch.int32), _dev_ptr(weights, "weights", torch.float32),
                                     _stream_on(dev, stream)), "mr_route_topk")
    return ids, weights


def moe_sort(topk_ids, num_experts: int, block: int, out=None, scratch: Scratch | None = None,
             stream=None):
    """(sorted_token_ids [cap], expert_ids [cap/block], num_tokens_post_padded [1]) int32."""
    torch = _torch()
    st0, ex0, nt0 = out if out is not None else (None, None, None)
    dev = _one_device(topk_ids=topk_ids, sorted_token_ids=st0, expert_ids=ex0, num_tokens_post_padded=nt0)
    if topk_ids.dim() != 2 or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be contiguous [M, k]")
    M, k = topk_ids.shape
    cap = sort_capacity(M, k, num_experts, block)
    if cap < 0:
        raise MoeRouteUnsupported(MR_ERR_UNSUPPORTED, "mr_sort_capacity")
    if out is None:
        out = (torch.empty(cap, dtype=torch.int32, device=dev),
               torch.empty(cap // block, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    st, ex, nt = out
    _check_sort_out(st, ex, nt, cap, block, dev)
    _check_scratch(scratch, dev)
    sp, sb = (scratch.ptr, scratch.nbytes) if scratch is not None else (None, 0)
    if scratch is None and M * k > PSORT_MAX_ASSIGN:
        scratch = Scratch(M, num_experts, 512, k, device=dev)
        sp, sb = scratch.ptr, scratch.nbytes
    with _launch_ctx(dev):
        _check(_load().mr_moe_sort(_dev_ptr(topk_ids, "topk_ids", torch.int32), M, k, num_experts, block,
                                   _dev_ptr(st, "sorted_token_ids", torch.int32),
                                   _dev_ptr(ex, "expert_ids", torch.int32),
                                   _dev_ptr(nt, "num_tokens_post_padded", torch.int32), st.numel(), sp, sb,
                                   _stream_on(dev, stream)), "mr_moe_sort")
    return st, ex, nt


def _check_sort_out(st, ex, nt, cap, block, dev):
    """The sort's outputs: st holds at least the capacity (its length is the
    capacity passed on), ex one entry per block of it, nt one entry."""
    torch = _torch()
    _check_out(st, "sorted_token_ids", cap, torch.int32, dev, min_numel=True)
    _check_out(ex, "expert_ids", st.numel() // block, torch.int32, dev, min_numel=True)
    _check_out(nt, "num_tokens_post_padded", 1, torch.int32, dev, min_numel=True)


def mxfp8_quant(x, out=None, stream=None):
    """(q uint8 [M, K] e4m3 codes, scale uint8 [M, K/32] e8m0)."""
    return _mx_quant(x, out, stream, fp4=False)


def _mx_quant(x, out, stream, fp4):
    torch = _torch()
    dev = _one_device(x=x, **({} if out is None else dict(q=out[0], scale=out[1])))
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    qk = K // 2 if fp4 else K
    if out is None:
        out = (torch.empty((M, qk), dtype=torch.uint8, device=dev),
               torch.empty((M, K // 32), dtype=torch.uint8, device=dev))
    q, s = out
    _check_out(q, "q", (M, qk), torch.uint8, dev)
    _check_out(s, "scale", (M, K // 32), torch.uint8, dev)
    fn, name = (_load().mr_mxfp4_quant, "mr_mxfp4_quant") if fp4 else (_load().mr_mxfp8_quant, "mr_mxfp8_quant")
    with _launch_ctx(dev):
        _check(fn(_dev_ptr(x, "x", torch.bfloat16), ldx, M, K, _dev_ptr(q, "q", torch.uint8),
                  _dev_ptr(s, "scale", torch.uint8), _stream_on(dev, stream)), name)
    return q, s


def route_output_layout(M: int, N: int, K: int, topk: int, block: int, quant=True):
    """[(name, dtype, shape, byte offset)] of the one-launch route's outputs
    packed into one buffer (each 16-byte aligned), and the buffer's bytes."""
    torch = _torch()
    cap = sort_capacity(M, topk, N, block)
    items = [("logits", torch.float32, (M, N)), ("topk_ids", torch.int32, (M, topk)),
             ("topk_weights", torch.float32, (M, topk)), ("sorted_token_ids", torch.int32, (cap,)),
             ("expert_ids", torch.int32, (cap // block,)), ("num_tokens_post_padded", torch.int32, (1,))]
    if quant:
        items += [("q", torch.uint8, (M, K // 2 if quant == "mxfp4" else K)), ("scale", torch.uint8, (M, K // 32))]
    layout, off = [], 0
    for name, dt, shape in items:
        n = 1
        for d in shape:
            n *= d
        layout.append((name, dt, shape, off))
        off += (n * torch.tensor([], dtype=dt).element_size() + 15) // 16 * 16
    return layout, off


def route_outputs_in(buf, M: int, N: int, K: int, topk: int, block: int, quant=True, offset: int = 0):
    """Views of the route's outputs inside the uint8 buffer buf, from byte
    offset (16-byte aligned) on: one copy of buf moves every output."""
    layout, nbytes = route_output_layout(M, N, K, topk, block, quant)
    if offset % 16 or buf.dtype != _torch().uint8 or buf.numel() < offset + nbytes:
        raise ValueError("buf must be uint8 with room for the outputs at a 16-byte aligned offset")
    out = {}
    for name, dt, shape, off in layout:
        n = 1
        for d in shape:
            n *= d
        esz = _torch().tensor([], dtype=dt).element_size()
        out[name] = buf[offset + off: offset + off + n * esz].view(dt).view(shape)
    return out


def mxfp4_quant(x, out=None, stream=None):
    """(q uint8 [M, K/2] packed e2m1 codes, element 2j in the low nibble;
    scale uint8 [M, K/32] e8m0)."""
    return _mx_quant(x, out, stream, fp4=True)


def alloc_route_outputs(M: int, N: int, K: int, topk: int, block: int, device, quant=True):
    """Output tensors of the one-launch route (a dict).  quant: True or
    "mxfp8" (q [M, K]), "mxfp4" (q [M, K/2]), False or None (no q / scale)."""
    torch = _torch()
    cap = sort_capacity(M, topk, N, block)
    out = dict(
        logits=torch.empty((M, N), dtype=torch.float32, device=device),
        topk_ids=torch.empty((M, topk), dtype=torch.int32, device=device),
        topk_weights=torch.empty((M, topk), dtype=torch.float32, device=device),
        sorted_token_ids=torch.empty(cap, dtype=torch.int32, device=device),
        expert_ids=torch.empty(cap // block, dtype=torch.int32, device=device),
        num_tokens_post_padded=torch.empty(1, dtype=torch.int32, device=device),
    )
    if quant:
        out["q"] = torch.empty((M, K // 2 if quant == "mxfp4" else K), dtype=torch.uint8, device=device)
        out["scale"] = torch.empty((M, K // 32), dtype=torch.uint8, device=device)
    return out


def _check_route_out(out, M, N, K, topk, block, quant, dev):
    """Every output of the one-launch route: dtype, shape (the sort's at
    least the capacity), contiguity and device."""
    torch = _torch()
    cap = sort_capacity(M, topk, N, block)
    if cap < 0:
        raise MoeRouteUnsupported(MR_ERR_UNSUPPORTED, "mr_sort_capacity")
    _check_out(out["logits"], "logits", (M, N), torch.float32, dev)
    _check_out(out["topk_ids"], "topk_ids", (M, topk), torch.int32, dev)
    _check_out(out["topk_weights"], "topk_weights", (M, topk), torch.float32, dev)
    _check_sort_out(out["sorted_token_ids"], out["expert_ids"], out["num_tokens_post_padded"], cap, block, dev)
    if quant:
        _check_out(out["q"], "q", (M, K // 2 if quant == "mxfp4" else K), torch.uint8, dev)
        _check_out(out["scale"], "scale", (M, K // 32), torch.uint8, dev)


def _check_w(w, K):
    if w.dim() != 2 or not w.is_contiguous() or w.shape[1] != K:
        raise ValueError("w must be contiguous [N, K]")


def _check_bias(bias, N, dev):
    if bias is not None:
        _check_out(bias, "bias", (N,), _torch().float32, dev)


def moe_route_sort_quant(x, w, topk: int, block: int, scoring: str = "softmax", bias=None,
                         renormalize: bool = True, quant: bool = True, out=None,
                         scratch: Scratch | None = None, stream=None):
    """The whole path for M <= 64 tokens in one launch; returns a dict of outputs."""
    torch = _torch()
    dev = _one_device(x=x, w=w, bias=bias)
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    N = w.shape[0]
    _check_w(w, K)
    _check_bias(bias, N, dev)
    if out is None:
        out = alloc_route_outputs(M, N, K, topk, block, dev, quant)
    _check_route_out(out, M, N, K, topk, block, quant, dev)
    if scratch is None:
        scratch = Scratch(M, N, K, topk, device=dev)
    _check_scratch(scratch, dev)
    q = out.get("q") if quant else None
    s = out.get("scale") if quant else None
    with _launch_ctx(dev):
        st = _load().mr_moe_route_sort_quant(
        _dev_ptr(x, "x", torch.bfloat16), ldx, _dev_ptr(w, "w", torch.bfloat16), M, N, K, topk,
        SCORING[scoring], _dev_ptr(bias, "bias", torch.float32, allow_none=True), int(renormalize), block,
        _dev_ptr(out["logits"], "logits", torch.float32), _dev_ptr(out["topk_ids"], "topk_ids", torch.int32),
        _dev_ptr(out["topk_weights"], "topk_weights", torch.float32),
        _dev_ptr(out["sorted_token_ids"], "sorted_token_ids", torch.int32),
        _dev_ptr(out["expert_ids"], "expert_ids", torch.int32),
        _dev_ptr(out["num_tokens_post_padded"], "num_tokens_post_padded", torch.int32),
        out["sorted_token_ids"].numel(), _dev_ptr(q, "q", torch.uint8, allow_none=True),
        _dev_ptr(s, "scale", torch.uint8, allow_none=True), scratch.ptr, scratch.nbytes,
        _stream_on(dev, stream))
    _check(st, "mr_moe_route_sort_quant")
    return out


def norm_apply(sres, rstd, norm_weight, norm: str = "gemma", out=None, stream=None):
    """The router input on the norm's scale, written out: bf16 [M, K] with
    xn[m, k] = bf16((sres[m, k] * rstd[m]) * s[k]), s = g or 1 + g."""
    torch = _torch()
    dev = _one_device(sres=sres, rstd=rstd, norm_weight=norm_weight, out=out)
    ldx = _row_major_2d(sres, "sres")
    M, K = sres.shape
    _check_norm_args(rstd, norm_weight, M, K)
    if out is None:
        out = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    _check_out(out, "out", (M, K), torch.bfloat16, dev)
    with _launch_ctx(dev):
        _check(_load().mr_norm_apply(_dev_ptr(sres, "sres", torch.bfloat16), ldx,
                                     _dev_ptr(rstd, "rstd", torch.float32),
                                     _dev_ptr(norm_weight, "norm_weight", torch.bfloat16), NORM_KIND[norm], M, K,
                                     _dev_ptr(out, "out", torch.bfloat16), _stream_on(dev, stream)),
               "mr_norm_apply")
    return out


def _check_norm_args(rstd, norm_weight, M, K):
    if rstd.dim() != 1 or rstd.shape[0] != M or not rstd.is_contiguous():
        raise ValueError("rstd must be contiguous [M]")
    if norm_weight.dim() != 1 or norm_weight.shape[0] != K or not norm_weight.is_contiguous():
        raise ValueError("norm_weight must be contiguous [K]")


def moe_route_sort_quant_norm(sres, rstd, norm_weight, w, topk: int, block: int, norm: str = "gemma",
                              scoring: str = "softmax", bias=None, renormalize: bool = True, quant: bool = True,
                              out=None, scratch: Scratch | None = None, stream=None):
    """The one-launch route with its input on the norm's scale (residual rows,
    per-token rstd, norm weight); returns a dict of outputs."""
    torch = _torch()
    dev = _one_device(sres=sres, rstd=rstd, norm_weight=norm_weight, w=w, bias=bias)
    ldx = _row_major_2d(sres, "sres")
    M, K = sres.shape
    N = w.shape[0]
    _check_w(w, K)
    _check_bias(bias, N, dev)
    _check_norm_args(rstd, norm_weight, M, K)
    if out is None:
        out = alloc_route_outputs(M, N, K, topk, block, dev, quant)
    _check_route_out(out, M, N, K, topk, block, quant, dev)
    if scratch is None:
        scratch = Scratch(M, N, K, topk, device=dev)
    _check_scratch(scratch, dev)
    q = out.get("q") if quant else None
    s = out.get("scale") if quant else None
    with _launch_ctx(dev):
        st = _load().mr_moe_route_sort_quant_norm(
        _dev_ptr(sres, "sres", torch.bfloat16), ldx, _dev_ptr(rstd, "rstd", torch.float32),
        _dev_ptr(norm_weight, "norm_weight", torch.bfloat16), NORM_KIND[norm],
        _dev_ptr(w, "w", torch.bfloat16), M, N, K, topk,
        SCORING[scoring], _dev_ptr(bias, "bias", torch.float32, allow_none=True), int(renormalize), block,
        _dev_ptr(out["logits"], "logits", torch.float32), _dev_ptr(out["topk_ids"], "topk_ids", torch.int32),
        _dev_ptr(out["topk_weights"], "topk_weights", torch.float32),
        _dev_ptr(out["sorted_token_ids"], "sorted_token_ids", torch.int32),
        _dev_ptr(out["expert_ids"], "expert_ids", torch.int32),
        _dev_ptr(out["num_tokens_post_padded"], "num_tokens_post_padded", torch.int32),
        out["sorted_token_ids"].numel(), _dev_ptr(q, "q", torch.uint8, allow_none=True),
        _dev_ptr(s, "scale", torch.uint8, allow_none=True), scratch.ptr, scratch.nbytes,
        _stream_on(dev, stream))
    _check(st, "mr_moe_route_sort_quant_norm")
    return out


class RouteParams(ctypes.Structure):
    """mr_route_params of moe_route.h, field for field."""
    _fields_ = [
        ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("rstd", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p), ("norm_kind", ctypes.c_int), ("w", ctypes.c_void_p),
        ("M", ctypes.c_int), ("N", ctypes.c_int), ("K", ctypes.c_int), ("topk", ctypes.c_int),
        ("scoring", ctypes.c_int), ("sel_bias", ctypes.c_void_p), ("renormalize", ctypes.c_int),
        ("block", ctypes.c_int), ("quant_format", ctypes.c_int), ("logits", ctypes.c_void_p),
        ("topk_ids", ctypes.c_void_p), ("topk_weights", ctypes.c_void_p), ("sorted_token_ids", ctypes.c_void_p),
        ("expert_ids", ctypes.c_void_p), ("num_tokens_post_padded", ctypes.c_void_p), ("capacity", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("scratch", ctypes.c_void_p),
        ("scratch_bytes", ctypes.c_size_t), ("shared_w13", ctypes.c_void_p), ("shared_w13_scale", ctypes.c_void_p),
        ("shared_inter", ctypes.c_int), ("shared_act", ctypes.c_void_p),
    ]


def moe_route(x, w, topk: int, block: int, scoring: str = "softmax", bias=None, renormalize: bool = True,
              quant="mxfp8", rstd=None, norm_weight=None, norm: str = "gemma", out=None,
              scratch: Scratch | None = None, stream=None, shared=None):
    """The one-launch route with every option (mr_moe_route): quant "mxfp8",
    "mxfp4" or None; with rstd (and norm_weight) x holds the residual rows
    and the route runs on the norm's scale; shared = (w13 E4M3 codes [2I, K],
    scale bytes [2I, K/32]) adds the shared expert's gate/up + SwiGLU to the
    launch (out["shared_act"], bf16 [M, I]).  Returns a dict of outputs."""
    call = PreparedRoute(x, w, topk, block, scoring, bias, renormalize, quant, rstd, norm_weight, norm, out, scratch,
                         shared)
    call(stream)
    return call.out


def _check_shared(shared, M, K, dev):
    """(w13, w13_scale) of the shared expert: uint8 [2I, K] and [2I, K/32]; returns I."""
    torch = _torch()
    w13, sc = shared
    if w13.dim() != 2 or w13.shape[1] != K or w13.shape[0] % 2:
        raise ValueError("w13 must be [2I, K]")
    R = w13.shape[0]
    _check_out(w13, "w13", (R, K), torch.uint8, dev)
    _check_out(sc, "w13_scale", (R, K // 32), torch.uint8, dev)
    return R // 2


def shared_gate_up(x, w13, w13_scale, out=None, stream=None):
    """The shared expert's gate/up projection and SwiGLU (mr_shared_gate_up):
    bf16 [M, I] = silu(x . gate^T) * (x . up^T) with MXFP8 w13 (E4M3 codes
    [2I, K], gate rows first, E8M0 scales [2I, K/32]); M <= 16."""
    torch = _torch()
    dev = _one_device(x=x, w13=w13, w13_scale=w13_scale, out=out)
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    I = _check_shared((w13, w13_scale), M, K, dev)
    if out is None:
        out = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
    _check_out(out, "out", (M, I), torch.bfloat16, dev)
    with _launch_ctx(dev):
        _check(_load().mr_shared_gate_up(_dev_ptr(x, "x", torch.bfloat16), ldx, _dev_ptr(w13, "w13", torch.uint8),
                                         _dev_ptr(w13_scale, "w13_scale", torch.uint8), M, K, I,
                                         _dev_ptr(out, "out", torch.bfloat16), _stream_on(dev, stream)),
               "mr_shared_gate_up")
    return out


class PreparedRoute:
    """The one-launch route over fixed buffers: the arguments are checked and
    the mr_route_params block is built once; each call is one launch of
    mr_moe_route on the given (or torch's current) stream.  The tensors are
    referenced for the object's life; refill x (and rstd) in place between
    calls.  Arguments as moe_route."""

    def __init__(self, x, w, topk: int, block: int, scoring: str = "softmax", bias=None, renormalize: bool = True,
                 quant="mxfp8", rstd=None, norm_weight=None, norm: str = "gemma", out=None,
                 scratch: Scratch | None = None, shared=None):
        self.p, self.out, self._keep = _route_params(x, w, topk, block, scoring, bias, renormalize, quant, rstd,
                                                     norm_weight, norm, out, scratch, shared)
        self.device = x.device
        self._ref = ctypes.byref(self.p)
        self._fn = _load().mr_moe_route

    def __call__(self, stream=None):
        """Launch on the route's device; stream: a torch stream of that
        device, a raw cudaStream_t (int) of that device, or None (torch's
        current stream there)."""
        torch = _torch()
        if isinstance(stream, int):
            sp = stream
        else:
            if stream is not None and stream.device != self.device:
                raise ValueError(f"stream must be on {self.device}")
            sp = _stream_on(self.device, stream)
        if torch.cuda.current_device() == self.device.index:
            status = self._fn(self._ref, sp)
        else:
            with _launch_ctx(self.device):
                status = self._fn(self._ref, sp)
        if status != MR_OK:
            _check(status, "mr_moe_route")
        return self.out


def _route_params(x, w, topk, block, scoring, bias, renormalize, quant, rstd, norm_weight, norm, out, scratch,
                  shared=None):
    torch = _torch()
    ldx = _row_major_2d(x, "x")
    M, K = x.shape
    N = w.shape[0]
    _check_w(w, K)
    if quant not in QUANT_FORMAT:
        raise ValueError(f"quant must be one of {list(QUANT_FORMAT)}")
    if rstd is not None:
        if norm_weight is None:
            raise ValueError("rstd needs norm_weight")
        _check_norm_args(rstd, norm_weight, M, K)
    dev = _one_device(x=x, w=w, bias=bias, rstd=rstd, norm_weight=norm_weight)
    _check_bias(bias, N, dev)
    if out is None:
        out = alloc_route_outputs(M, N, K, topk, block, dev, quant)
    _check_route_out(out, M, N, K, topk, block, quant, dev)
    if scratch is None:
        scratch = Scratch(M, N, K, topk, device=dev)
    _check_scratch(scratch, dev)
    p = RouteParams()
    p.x = _dev_ptr(x, "x", torch.bfloat16)
    p.ldx = ldx
    p.rstd = _dev_ptr(rstd, "rstd", torch.float32, allow_none=True)
    p.norm_weight = _dev_ptr(norm_weight, "norm_weight", torch.bfloat16, allow_none=True)
    p.norm_kind = NORM_KIND[norm]
    p.w = _dev_ptr(w, "w", torch.bfloat16)
    p.M, p.N, p.K, p.topk = M, N, K, topk
    p.scoring = SCORING[scoring]
    p.sel_bias = _dev_ptr(bias, "bias", torch.float32, allow_none=True)
    p.renormalize = int(renormalize)
    p.block = block
    p.quant_format = QUANT_FORMAT[quant]
    p.logits = _dev_ptr(out["logits"], "logits", torch.float32)
    p.topk_ids = _dev_ptr(out["topk_ids"], "topk_ids", torch.int32)
    p.topk_weights = _dev_ptr(out["topk_weights"], "topk_weights", torch.float32)
    p.sorted_token_ids = _dev_ptr(out["sorted_token_ids"], "sorted_token_ids", torch.int32)
    p.expert_ids = _dev_ptr(out["expert_ids"], "expert_ids", torch.int32)
    p.num_tokens_post_padded = _dev_ptr(out["num_tokens_post_padded"], "num_tokens_post_padded", torch.int32)
    p.capacity = out["sorted_token_ids"].numel()
    if quant is not None:
        qt, st = out["q"], out["scale"]
        p.q = _dev_ptr(qt, "q", torch.uint8)
        p.scale = _dev_ptr(st, "scale", torch.uint8)
    p.scratch = scratch.ptr
    p.scratch_bytes = scratch.nbytes
    if shared is not None:
        I = _check_shared(shared, M, K, dev)
        if "shared_act" not in out:
            out["shared_act"] = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
        _check_out(out["shared_act"], "shared_act", (M, I), torch.bfloat16, dev)
        p.shared_w13 = _dev_ptr(shared[0], "w13", torch.uint8)
        p.shared_w13_scale = _dev_ptr(shared[1], "w13_scale", torch.uint8)
        p.shared_inter = I
        p.shared_act = _dev_ptr(out["shared_act"], "shared_act", torch.bfloat16)
    return p, out, (x, w, bias, rstd, norm_weight, scratch, shared)


def moe_sort_quant(topk_ids, x, num_experts: int, block: int, quant: str = "mxfp8", out=None, stream=None,
                   sorted_rows: bool = False):
    """Sort and stage-1 quant in one launch (decode batches, M * topk <= 65536):
    (sorted_token_ids, expert_ids, num_tokens_post_padded, q, scale).  q and
    scale are in token order ([M, K or K/2], [M, K/32]), or with sorted_rows
    in sorted order ([capacity, ...] rows: row p quantises the token of the
    assignment at sorted position p, padding rows are zero, rows past
    num_tokens_post_padded are left as they were)."""
    torch = _torch()
    if topk_ids.dim() != 2 or not topk_ids.is_contiguous():
        raise ValueError("topk_ids must be contiguous [M, k]")
    M, k = topk_ids.shape
    ldx = _row_major_2d(x, "x")
    if x.shape[0] != M:
        raise ValueError("x must have the rows of topk_ids")
    K = x.shape[1]
    if quant not in ("mxfp8", "mxfp4"):
        raise ValueError("quant must be mxfp8 or mxfp4")
    dev = _one_device(topk_ids=topk_ids, x=x)
    cap = sort_capacity(M, k, num_experts, block)
    if cap < 0:
        raise MoeRouteUnsupported(MR_ERR_UNSUPPORTED, "mr_sort_capacity")
    rows = cap if sorted_rows else M
    qk = K // 2 if quant == "mxfp4" else K
    if out is None:
        out = (torch.empty(cap, dtype=torch.int32, device=dev), torch.empty(cap // block, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev), torch.empty((rows, qk), dtype=torch.uint8, device=dev),
               torch.empty((rows, K // 32), dtype=torch.uint8, device=dev))
    st, ex, nt, q, s = out
    _check_sort_out(st, ex, nt, cap, block, dev)
    if sorted_rows and st.numel() != cap:
        raise ValueError("sorted rows: sorted_token_ids must hold exactly the capacity (its rows index q)")
    _check_out(q, "q", (rows, qk), torch.uint8, dev)
    _check_out(s, "scale", (rows, K // 32), torch.uint8, dev)
    fmt = QUANT_FORMAT[quant] | (QUANT_SORTED_ROWS if sorted_rows else 0)
    with _launch_ctx(dev):
        status = _load().mr_moe_sort_quant(_dev_ptr(topk_ids, "topk_ids", torch.int32), M, k, num_experts, block,
                                           _dev_ptr(x, "x", torch.bfloat16), ldx, K, fmt,
                                           _dev_ptr(st, "sorted_token_ids", torch.int32),
                                           _dev_ptr(ex, "expert_ids", torch.int32),
                                           _dev_ptr(nt, "num_tokens_post_padded", torch.int32), st.numel(),
                                           _dev_ptr(q, "q", torch.uint8), _dev_ptr(s, "scale", torch.uint8),
                                           _stream_on(dev, stream))
    _check(status, "mr_moe_sort_quant")
    return st, ex, nt, q, s
