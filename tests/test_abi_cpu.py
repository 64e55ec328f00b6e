"""The C ABI library on a machine without a GPU: it builds, loads, exports
every entry point include/moe_route.h declares, and its host-only functions
(shape predicate, sizes, validation) behave.  No call here reaches a kernel."""

import ctypes
import os
import re
import subprocess

import pytest

import decode_expert_routing_gb300 as mr
from decode_expert_routing_gb300 import build as mrbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_route.h")


@pytest.fixture(scope="module")
def lib():
    mrbuild.build()
    return mr.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mr_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("mr_router_gemv", "mr_route_topk", "mr_moe_sort", "mr_mxfp8_quant",
              "mr_moe_route_sort_quant", "mr_router_gemv_supported", "mr_scratch_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(mr.SIGNATURES), "binding signatures out of sync with the header"
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.mr_abi_version() == 2
    for s in range(7):
        assert lib.mr_status_string(s).startswith(b"MR_")
    assert b"SCRATCH_DIRTY" in lib.mr_status_string(mr.MR_ERR_SCRATCH_DIRTY)
    assert lib.mr_status_string(99) == b"unknown mr_status"
    assert lib.mr_last_cuda_error() == 0  # no call of this thread has returned MR_ERR_CUDA


def test_shape_predicate(lib):
    ok = mr.router_gemv_supported
    assert ok(1, 128, 6144) and ok(16, 128, 6144) and ok(64, 128, 6144) and ok(512, 128, 6144)
    assert ok(8, 896, 3584) and ok(32, 896, 3584)
    assert not ok(513, 128, 6144)          # M > 512
    assert not ok(1, 128, 6000)            # K % 512
    assert not ok(1, 100, 6144)            # N % 8
    assert not ok(100, 100, 6144)          # N % BLOCK_N of the split-K GEMV
    assert not ok(1, 2048, 6144)           # N > 1024
    assert not ok(0, 128, 6144)
    assert not ok(1, 128, 6144, 6143)      # ldx < K
    assert not ok(1, 128, 6144, 6148)      # ldx % 8
    assert ok(1, 128, 6144, 6144 + 64)


def test_sort_capacity(lib):
    assert mr.sort_capacity(1, 8, 128, 16) == 128
    assert mr.sort_capacity(3, 2, 4, 2) == 10
    assert mr.sort_capacity(32, 16, 896, 16) == 512 + 512 * 15
    assert mr.sort_capacity(4096, 8, 128, 64) == 32768 + 128 * 63
    assert mr.sort_capacity(0, 8, 128, 16) == -1


def test_scratch_bytes(lib):
    b = mr.scratch_bytes(64, 128, 6144, 8)
    assert b >= 32768 and b % 256 == 0
    # covers the largest split-K partial plane of any M up to M_max, and the
    # tensor-core GEMV's partials ((M + 127) rows x N x 16 slices of fp32 at most)
    assert mr.scratch_bytes(512, 128, 6144, 8) >= 32768 + (512 + 127) * 128 * 16 * 4
    assert mr.scratch_bytes(65, 128, 6144, 8) >= 32768 + (65 + 127) * 128 * 16 * 4
    assert mr.scratch_bytes(512, 128, 6144, 8) >= b
    assert mr.scratch_bytes(4096, 128, 6144, 8) >= 32768 + 4 * 32768
    assert mr.scratch_bytes(0, 128, 6144, 8) == 0
    # the fused route over several clusters gathers every token's ids
    assert mr.scratch_bytes(64, 1024, 512, 32) >= 32768 + 64 * 32 * 4


def test_validation_returns_before_any_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    # null x
    assert lib.mr_router_gemv(None, 6144, fake, fake, 1, 128, 6144, fake, 1 << 20, None) == mr.MR_ERR_INVALID_ARG
    # misaligned x
    assert lib.mr_router_gemv(P(0x1002), 6144, fake, fake, 1, 128, 6144, fake, 1 << 20, None) == mr.MR_ERR_INVALID_ARG
    # unsupported K
    assert lib.mr_router_gemv(fake, 6000, fake, fake, 1, 128, 6000, fake, 1 << 20, None) == mr.MR_ERR_UNSUPPORTED
    # scratch too small (above 64 rows, a shape the cluster kernel does not
    # hold in shared memory goes to the split-K GEMV, which needs scratch)
    assert lib.mr_router_gemv(fake, 6144, fake, fake, 100, 1024, 6144, fake, 100, None) == mr.MR_ERR_SCRATCH_TOO_SMALL
    assert lib.mr_router_gemv(fake, 6144, fake, fake, 100, 1024, 6144, None, 0, None) == mr.MR_ERR_INVALID_ARG
    # gate: topk > N, bad scoring, N too large
    assert lib.mr_route_topk(fake, 1, 8, 9, 0, None, 1, fake, fake, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_route_topk(fake, 1, 128, 8, 7, None, 1, fake, fake, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_route_topk(fake, 1, 2048, 8, 0, None, 1, fake, fake, None) == mr.MR_ERR_UNSUPPORTED
    assert lib.mr_route_topk(fake, 1, 128, 33, 0, None, 1, fake, fake, None) == mr.MR_ERR_UNSUPPORTED
    # sort: capacity too small
    assert lib.mr_moe_sort(fake, 1, 8, 128, 16, fake, fake, fake, 64, None, 0, None) == mr.MR_ERR_INVALID_ARG
    # sort of a large batch without scratch
    assert mr.sort_capacity(9000, 8, 128, 64) == 80064
    assert lib.mr_moe_sort(fake, 9000, 8, 128, 64, fake, fake, fake, 80064, None, 0, None) == mr.MR_ERR_INVALID_ARG
    # quant: K % 32
    assert lib.mr_mxfp8_quant(fake, 48, 1, 40, fake, fake, None) == mr.MR_ERR_UNSUPPORTED
    # fused: M > 64
    assert lib.mr_moe_route_sort_quant(fake, 6144, fake, 65, 128, 6144, 8, 0, None, 1, 16, fake, fake, fake,
                                       fake, fake, fake, 1 << 20, fake, fake, fake, 1 << 20, None) == mr.MR_ERR_UNSUPPORTED
    # fused: q without scale
    assert lib.mr_moe_route_sort_quant(fake, 6144, fake, 1, 128, 6144, 8, 0, None, 1, 16, fake, fake, fake,
                                       fake, fake, fake, 128, fake, None, fake, 1 << 20, None) == mr.MR_ERR_INVALID_ARG
    # fused over several clusters (M > 16): the ticket and the ids live in scratch
    assert lib.mr_moe_route_sort_quant(fake, 6144, fake, 17, 128, 6144, 8, 0, None, 1, 16, fake, fake, fake,
                                       fake, fake, fake, 1 << 20, fake, fake, None, 0, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_moe_route_sort_quant(fake, 6144, fake, 17, 128, 6144, 8, 0, None, 1, 16, fake, fake, fake,
                                       fake, fake, fake, 1 << 20, fake, fake, fake, 32768 + 17 * 8 * 4 - 4,
                                       None) == mr.MR_ERR_SCRATCH_TOO_SMALL
    # route on the norm's scale: null rstd, misaligned norm weight, unknown
    # norm kind; then the fused route's own checks (M > 64)
    args = (fake, 128, 6144, 8, 0, None, 1, 16, fake, fake, fake, fake, fake, fake, 1 << 20, fake, fake, fake,
            1 << 20, None)
    assert lib.mr_moe_route_sort_quant_norm(fake, 6144, None, fake, 1, fake, 1, *args[1:]) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_moe_route_sort_quant_norm(fake, 6144, fake, P(0x1008), 1, fake, 1,
                                            *args[1:]) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_moe_route_sort_quant_norm(fake, 6144, fake, fake, 2, fake, 1, *args[1:]) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_moe_route_sort_quant_norm(fake, 6144, fake, fake, 1, fake, 65, *args[1:]) == mr.MR_ERR_UNSUPPORTED
    # written-out norm: K % 8, null output, bad kind
    assert lib.mr_norm_apply(fake, 48, fake, fake, 0, 2, 44, fake, None) == mr.MR_ERR_UNSUPPORTED
    assert lib.mr_norm_apply(fake, 48, fake, fake, 0, 2, 48, None, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_norm_apply(fake, 48, fake, fake, 5, 2, 48, fake, None) == mr.MR_ERR_INVALID_ARG
    # launch options and the wait limit (host-only settings)
    assert lib.mr_set_launch_flags(32) == mr.MR_ERR_INVALID_ARG
    for f in (mr.LAUNCH_TEST_SLOW_SIGMOID, mr.LAUNCH_CHECK_SCRATCH):
        assert lib.mr_set_launch_flags(f) == mr.MR_OK and lib.mr_get_launch_flags() == f
    assert lib.mr_set_launch_flags(mr.LAUNCH_LEGACY_MMA) == mr.MR_OK
    assert lib.mr_get_launch_flags() == mr.LAUNCH_LEGACY_MMA
    assert lib.mr_set_launch_flags(0) == mr.MR_OK
    assert lib.mr_set_wait_limit_ns(999) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_set_wait_limit_ns(60_000_000_001) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_set_wait_limit_ns(1_000_000_000) == mr.MR_OK
    # reset: buffer below the counter prefix
    assert lib.mr_scratch_reset(fake, 100, None) == mr.MR_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    saved = mr._lib
    try:
        mr._lib = None
        with pytest.raises(RuntimeError, match="not found"):
            mr.load_library(str(tmp_path / "nope.so"))
    finally:
        mr._lib = saved


def test_route_params_layout_matches_header(tmp_path):
    # compile a probe against the header with the host C compiler and compare
    # every field offset and the size with the binding's ctypes structure
    fields = [f for f, _ in mr.RouteParams._fields_]
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moe_route.h"\nint main(void) {\n'
                   + "".join(f'  printf("%zu\\n", offsetof(mr_route_params, {f}));\n' for f in fields)
                   + '  printf("%zu\\n", sizeof(mr_route_params));\n  return 0;\n}\n')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    want = [getattr(mr.RouteParams, f).offset for f in fields] + [ctypes.sizeof(mr.RouteParams)]
    assert out == want


def test_general_route_and_mxfp4_validation(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.mr_moe_route(None, None) == mr.MR_ERR_INVALID_ARG
    p = mr.RouteParams()
    p.x, p.ldx, p.w = 0x1000, 6144, 0x1000
    p.M, p.N, p.K, p.topk, p.scoring, p.renormalize, p.block = 4, 128, 6144, 8, 0, 1, 16
    for f in ("logits", "topk_ids", "topk_weights", "sorted_token_ids", "expert_ids", "num_tokens_post_padded",
              "q", "scale"):
        setattr(p, f, 0x1000)
    p.capacity = 1 << 20
    p.quant_format = 7                       # unknown format
    assert lib.mr_moe_route(ctypes.byref(p), None) == mr.MR_ERR_INVALID_ARG
    p.quant_format = 2
    p.q = 0x1004                             # MXFP4 output must be 8-byte aligned here
    assert lib.mr_moe_route(ctypes.byref(p), None) == mr.MR_ERR_INVALID_ARG
    p.q = 0x1000
    p.M = 65                                 # the one launch covers M <= 64
    assert lib.mr_moe_route(ctypes.byref(p), None) == mr.MR_ERR_UNSUPPORTED
    p.M, p.rstd, p.norm_weight, p.norm_kind = 4, 0x1000, 0x1000, 3   # unknown norm kind
    assert lib.mr_moe_route(ctypes.byref(p), None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_mxfp4_quant(fake, 48, 1, 40, fake, fake, None) == mr.MR_ERR_UNSUPPORTED
    # sort + quant in one launch: too many assignments, no quant format, misaligned q
    assert lib.mr_moe_sort_quant(fake, 8193, 8, 128, 16, fake, 512, 512, 1, fake, fake, fake, 1 << 20, fake, fake,
                                 None) == mr.MR_ERR_UNSUPPORTED
    assert lib.mr_moe_sort_quant(fake, 4, 8, 128, 16, fake, 512, 512, 0, fake, fake, fake, 1 << 20, fake, fake,
                                 None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_moe_sort_quant(fake, 4, 8, 128, 16, fake, 512, 512, 2, fake, fake, fake, 1 << 20, P(0x1004), fake,
                                 None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_mxfp4_quant(fake, 64, 1, 64, P(0x1002), fake, None) == mr.MR_ERR_INVALID_ARG


def test_route_output_arena_layout():
    import torch
    for quant in (True, "mxfp4", None):
        layout, nbytes = mr.route_output_layout(16, 128, 6144, 8, 16, quant)
        names = [n for n, _, _, _ in layout]
        assert names[:6] == ["logits", "topk_ids", "topk_weights", "sorted_token_ids", "expert_ids",
                             "num_tokens_post_padded"]
        assert ("q" in names) == bool(quant)
        assert all(off % 16 == 0 for _, _, _, off in layout) and nbytes % 16 == 0
        buf = torch.zeros(nbytes + 32, dtype=torch.uint8)
        out = mr.route_outputs_in(buf, 16, 128, 6144, 8, 16, quant, offset=32)
        cap = mr.sort_capacity(16, 8, 128, 16)
        assert out["logits"].shape == (16, 128) and out["logits"].dtype == torch.float32
        assert out["sorted_token_ids"].shape == (cap,) and out["expert_ids"].shape == (cap // 16,)
        if quant:
            assert out["q"].shape == (16, 6144 // 2 if quant == "mxfp4" else 6144)
        # disjoint views inside the buffer
        spans = sorted((t.data_ptr() - buf.data_ptr(), t.numel() * t.element_size()) for t in out.values())
        assert spans[0][0] >= 32 and all(a + n <= b for (a, n), (b, _) in zip(spans, spans[1:]))
        assert spans[-1][0] + spans[-1][1] <= buf.numel()
    with pytest.raises(ValueError):
        mr.route_outputs_in(torch.zeros(64, dtype=torch.uint8), 16, 128, 6144, 8, 16)


def test_binding_rejects_bad_arguments_and_host_tensors():
    # argument checks run before any launch; host tensors are refused (there
    # is no CPU path behind the binding)
    import torch
    x = torch.zeros((4, 512), dtype=torch.bfloat16)
    w = torch.zeros((128, 512), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="quant"):
        mr.moe_route(x, w, 8, 16, quant="fp16")
    with pytest.raises(ValueError, match="norm_weight"):
        mr.moe_route(x, w, 8, 16, rstd=torch.ones(4))
    with pytest.raises(ValueError, match="rstd"):
        mr.moe_route(x, w, 8, 16, rstd=torch.ones(3), norm_weight=torch.zeros(512, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        mr.moe_route(x, w, 8, 16)
    with pytest.raises(ValueError, match="CUDA"):
        mr.mxfp4_quant(x)
    with pytest.raises(ValueError, match="CUDA"):
        mr.router_gemv(x, w)
    ids = torch.zeros((4, 8), dtype=torch.int32)
    with pytest.raises(ValueError, match="quant"):
        mr.moe_sort_quant(ids, x, 128, 16, quant="mxfp16")
    with pytest.raises(ValueError, match="rows"):
        mr.moe_sort_quant(ids, torch.zeros((5, 512), dtype=torch.bfloat16), 128, 16)
    with pytest.raises(ValueError, match="CUDA"):
        mr.moe_sort_quant(ids, x, 128, 16)


class _FakeCuda:
    """Stands in for a CUDA tensor in host-side argument checks (no GPU
    here): device, dtype, shape, strides and contiguity only.  Any use of
    its data would fail (data_ptr raises), so a check that lets a bad
    argument through to the library shows up as an error of the wrong kind."""

    def __init__(self, shape, dtype, device=0, contiguous=True):
        import torch
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device("cuda", device)
        self.is_cuda = True
        self._contig = contiguous

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for d in self.shape:
            n *= d
        return n

    def stride(self, i=None):
        st, acc = [], 1
        for d in reversed(self.shape):
            st.append(acc)
            acc *= d
        st = tuple(reversed(st))
        if not self._contig and len(st) == 2:
            st = (st[0] * 2, 1)
        return st if i is None else st[i]

    def is_contiguous(self):
        return self._contig

    def data_ptr(self):
        raise AssertionError("the library was reached with an argument the binding should have refused")


def test_binding_refuses_bad_outputs_and_mixed_devices():
    """Caller-passed outputs of the wrong shape, dtype or layout, and tensors
    on different devices, are refused before any launch (a short or strided
    output would be written out of bounds, a pointer of another device used
    on the current one)."""
    import torch
    bf, f32, i32, u8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8
    x, w = _FakeCuda((4, 512), bf), _FakeCuda((128, 512), bf)
    for fn in (mr.router_gemv, mr.router_gemv_noalloc):
        with pytest.raises(ValueError, match="shape"):
            fn(x, w, out=_FakeCuda((4, 64), f32))
        with pytest.raises(ValueError, match="contiguous"):
            fn(x, w, out=_FakeCuda((4, 128), f32, contiguous=False))
        with pytest.raises(ValueError, match="float32"):
            fn(x, w, out=_FakeCuda((4, 128), bf))
        with pytest.raises(ValueError, match="devices"):
            fn(x, _FakeCuda((128, 512), bf, device=1))
        with pytest.raises(ValueError, match="devices"):
            fn(x, w, out=_FakeCuda((4, 128), f32, device=1))
    lg = _FakeCuda((4, 128), f32)
    with pytest.raises(ValueError, match="ids"):
        mr.route_topk(lg, 8, ids=_FakeCuda((4, 4), i32), weights=_FakeCuda((4, 8), f32))
    with pytest.raises(ValueError, match="bias"):
        mr.route_topk(lg, 8, "sigmoid", bias=_FakeCuda((64,), f32),
                      ids=_FakeCuda((4, 8), i32), weights=_FakeCuda((4, 8), f32))
    cap = mr.sort_capacity(4, 8, 128, 16)
    ids = _FakeCuda((4, 8), i32)
    with pytest.raises(ValueError, match="sorted_token_ids"):
        mr.moe_sort(ids, 128, 16, out=(_FakeCuda((cap - 16,), i32), _FakeCuda((cap // 16,), i32), _FakeCuda((1,), i32)))
    with pytest.raises(ValueError, match="expert_ids"):
        mr.moe_sort(ids, 128, 16, out=(_FakeCuda((cap,), i32), _FakeCuda((cap // 16 - 1,), i32), _FakeCuda((1,), i32)))
    with pytest.raises(ValueError, match="q"):
        mr.mxfp8_quant(x, out=(_FakeCuda((4, 256), u8), _FakeCuda((4, 16), u8)))
    with pytest.raises(ValueError, match="q"):
        mr.mxfp4_quant(x, out=(_FakeCuda((4, 512), u8), _FakeCuda((4, 16), u8)))
    route_out = dict(logits=_FakeCuda((4, 128), f32), topk_ids=_FakeCuda((4, 8), i32),
                     topk_weights=_FakeCuda((4, 8), f32), sorted_token_ids=_FakeCuda((cap,), i32),
                     expert_ids=_FakeCuda((cap // 16,), i32), num_tokens_post_padded=_FakeCuda((1,), i32),
                     q=_FakeCuda((4, 512), u8), scale=_FakeCuda((4, 16), u8))
    for name, bad in (("logits", _FakeCuda((4, 127), f32)), ("topk_weights", _FakeCuda((4, 8), bf)),
                      ("q", _FakeCuda((4, 256), u8)), ("scale", _FakeCuda((4, 16), u8, device=1))):
        o = dict(route_out, **{name: bad})
        with pytest.raises(ValueError, match=name):
            mr.moe_route_sort_quant(x, w, 8, 16, out=o)
        with pytest.raises(ValueError, match=name):
            mr.moe_route(x, w, 8, 16, out=o)
    with pytest.raises(ValueError, match="devices"):
        mr.moe_route(x, w, 8, 16, out=route_out, bias=_FakeCuda((128,), f32, device=1), scoring="sigmoid")
    with pytest.raises(ValueError, match="scale"):
        mr.moe_sort_quant(ids, x, 128, 16, out=(_FakeCuda((cap,), i32), _FakeCuda((cap // 16,), i32),
                                                _FakeCuda((1,), i32), _FakeCuda((4, 512), u8),
                                                _FakeCuda((4, 8), u8)))
    with pytest.raises(ValueError, match="out"):
        mr.norm_apply(x, _FakeCuda((4,), f32), _FakeCuda((512,), bf), out=_FakeCuda((4, 256), bf))


def test_shared_gate_up_validation(lib):
    """Host checks of the shared expert's entry point (nothing launches)."""
    fake = ctypes.c_void_p(0x1000)
    P = ctypes.c_void_p
    # M above 16, K not a multiple of 512, I not a multiple of 8
    assert lib.mr_shared_gate_up(fake, 6144, fake, fake, 17, 6144, 768, fake, None) == mr.MR_ERR_UNSUPPORTED
    assert lib.mr_shared_gate_up(fake, 6144, fake, fake, 4, 6000, 768, fake, None) == mr.MR_ERR_UNSUPPORTED
    assert lib.mr_shared_gate_up(fake, 6144, fake, fake, 4, 6144, 100, fake, None) == mr.MR_ERR_UNSUPPORTED
    # null or misaligned weights / output
    assert lib.mr_shared_gate_up(fake, 6144, None, fake, 4, 6144, 768, fake, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_shared_gate_up(fake, 6144, P(0x1008), fake, 4, 6144, 768, fake, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_shared_gate_up(fake, 6144, fake, None, 4, 6144, 768, fake, None) == mr.MR_ERR_INVALID_ARG
    assert lib.mr_shared_gate_up(fake, 6144, fake, fake, 4, 6144, 768, P(0x1002), None) == mr.MR_ERR_INVALID_ARG
    # the route with a shared expert: more than 16 tokens is outside its cover
    p = mr.RouteParams()
    p.x, p.ldx, p.w, p.M, p.N, p.K, p.topk, p.block = fake, 6144, fake, 32, 128, 6144, 8, 16
    for f in ("logits", "topk_ids", "topk_weights", "sorted_token_ids", "expert_ids", "num_tokens_post_padded",
              "scratch", "shared_w13", "shared_w13_scale", "shared_act"):
        setattr(p, f, fake)
    p.capacity, p.scratch_bytes, p.shared_inter = 4096, 1 << 20, 768
    assert lib.mr_moe_route(ctypes.byref(p), None) == mr.MR_ERR_UNSUPPORTED
