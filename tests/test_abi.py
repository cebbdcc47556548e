"""CPU tests of the C ABI: the library builds, loads and exports every symbol
the header declares; host-side argument validation rejects bad calls with
the documented status before any CUDA call (the pointers used here are fake
and never dereferenced)."""
import ctypes
import os
import re

import pytest

from attention_all_layout_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_a2a.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bd.LIB_PATH):
        from attention_all_layout_gb300 import build

        build.build()
    return bd.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_expected_entry_points():
    assert header_functions() == sorted(bd.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_strerror(lib):
    assert bd.strerror(bd.OK) == "ok"
    assert "invalid" in bd.strerror(bd.EINVAL)
    assert "wait" in bd.strerror(bd.ETIMEOUT)
    assert bd.strerror(99) == "unknown status"


FAKE = 1 << 20  # 16-byte aligned, never dereferenced


def call_fwd(lib, B=1, H=4, S=256, d=64, P=2, scale=0.125, q=FAKE, k=FAKE * 2, v=FAKE * 3, parts=None,
             strides=None, opts=None):
    sb, sh, ss = H * S * d, S * d, d
    st = strides or (sb, sh, ss)
    shp = bd.Shape(B, H, S, d, *st, *st, *st)
    if parts is None:
        parts = [FAKE * (16 + j) for j in range(max(P, 1))]
    arr = (ctypes.c_void_p * max(1, len(parts)))(*parts)
    o = ctypes.byref(opts) if opts is not None else None
    return lib.attn_a2a_fwd_ex(q, k, v, ctypes.byref(shp), P, scale, arr, None, o, None)


@pytest.mark.parametrize(
    "kw,code",
    [
        (dict(P=0), bd.EINVAL),
        (dict(P=65, H=65), bd.EINVAL),
        (dict(P=3, H=4), bd.EINVAL),  # H % P != 0
        (dict(d=96), bd.EUNSUPPORTED),
        (dict(d=0), bd.EINVAL),
        (dict(scale=-1.0), bd.EINVAL),
        (dict(scale=float("nan")), bd.EINVAL),
        (dict(scale=float("inf")), bd.EINVAL),
        (dict(q=0), bd.EINVAL),
        (dict(k=FAKE + 8), bd.EINVAL),  # misaligned
        (dict(parts=[FAKE * 16, 0]), bd.EINVAL),  # null partition with rows
        (dict(parts=[FAKE * 16, FAKE * 17 + 2]), bd.EINVAL),  # misaligned partition
        (dict(strides=(4 * 256 * 64, 256 * 64, 60)), bd.EINVAL),  # sequence stride not a multiple of 8
        (dict(strides=(4 * 256 * 64, -256 * 64, 64)), bd.EINVAL),
        (dict(B=-1), bd.EINVAL),
        (dict(parts=[FAKE * 2, FAKE * 40]), bd.EINVAL),  # partition 0 aliases k
    ],
)
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert call_fwd(lib, **kw) == code


def test_bad_options_rejected(lib):
    assert call_fwd(lib, opts=bd._opts(store_kind=7)) == bd.EINVAL
    assert call_fwd(lib, opts=bd._opts(store_kind=4)) == bd.EINVAL
    # the bulk-store epilogue exists for the all-to-all layout with at most 8 partitions
    assert call_fwd(lib, P=16, H=16, opts=bd._opts(store_kind=1)) == bd.EUNSUPPORTED
    assert call_fwd(lib, opts=bd._opts(grid=-1)) == bd.EINVAL
    assert call_fwd(lib, opts=bd._opts(timeout_ns=-5)) == bd.EINVAL
    assert call_fwd(lib, opts=bd._opts(tile_order=2)) == bd.EINVAL
    assert call_fwd(lib, opts=bd._opts(cta_pairs=3)) == bd.EINVAL
    assert call_fwd(lib, opts=bd._opts(cta_pairs=-1)) == bd.EINVAL


def test_s2s_ex_options(lib):
    # the whole layer's entry point with options: what its kernels do not have
    # is refused before anything runs; out-of-range values are invalid
    shp = bd.plain_shape(1, 8, 4096, 128)
    parts = [FAKE * (16 + j) for j in range(8)]
    q, k, v = ([FAKE * (64 + 8 * i + j) for j in range(8)] for i in range(3))
    arr = lambda xs: (ctypes.c_void_p * 8)(*xs)

    def call(**kw):
        o = bd._opts(**kw)
        return lib.attn_a2a_fwd_s2s_ex(arr(q), arr(k), arr(v), ctypes.byref(shp), 8, 0.1, arr(parts), None,
                                       ctypes.byref(o), None)
    assert call(store_kind=3) == bd.EUNSUPPORTED
    assert call(tile_order=1) == bd.EUNSUPPORTED
    assert call(part_heads=16) == bd.EUNSUPPORTED
    assert call(cta_pairs=1) == bd.EUNSUPPORTED
    assert call(store_kind=4) == bd.EINVAL
    assert call(split=4) == bd.EINVAL
    assert call(grid=-1) == bd.EINVAL


def test_store_kind_query(lib):
    # the automatic kind: bulk tensor stores for the contiguous layout, and for
    # the all-to-all layout with P <= 8, at every length
    assert bd.attn_a2a_store_kind(32768, 1, 0) == 1
    assert bd.attn_a2a_store_kind(32768, 8, 1) == 1
    assert bd.attn_a2a_store_kind(32769, 8, 1) == 1
    assert bd.attn_a2a_store_kind(75600, 8, 1) == 1
    assert bd.attn_a2a_store_kind(4096, 16, 1) == 2
    assert bd.attn_a2a_store_kind(0, 2, 1) == 1
    # an explicit kind is kept where it is built
    assert bd.attn_a2a_store_kind(32768, 8, 1, store_kind=1) == 1
    assert bd.attn_a2a_store_kind(1024, 8, 1, store_kind=2) == 2
    # whole-line row stores: all-to-all layout only, never automatic
    assert bd.attn_a2a_store_kind(1024, 16, 1, store_kind=3) == 3
    out = ctypes.c_int(0)
    assert lib.attn_a2a_store_kind(4096, 16, 1, 1, ctypes.byref(out)) == bd.EUNSUPPORTED
    assert lib.attn_a2a_store_kind(4096, 1, 0, 3, ctypes.byref(out)) == bd.EUNSUPPORTED
    for args in ((4096, 8, 2, 0), (4096, 0, 1, 0), (4096, 65, 1, 0), (-1, 8, 1, 0), (4096, 8, 1, 4)):
        assert lib.attn_a2a_store_kind(*args, ctypes.byref(out)) == bd.EINVAL
    assert lib.attn_a2a_store_kind(4096, 8, 1, 0, None) == bd.EINVAL


def test_split_plan_query(lib):
    L2 = 126 * 2**20
    # image: the whole schedule in 81-block ranges; video: the last wave in 176-block ranges;
    # H = 40, S = 4096 (K and V beyond half of L2, tail saves too little): nothing
    assert bd.attn_a2a_split_plan(1, 24, 4096, 128, num_sms=152, l2_bytes=L2) == (bd.SPLIT_ALL, 0, 81)
    # joint: 103-block ranges would save 5 of 108 key blocks per CTA, too few
    assert bd.attn_a2a_split_plan(1, 24, 4608, 128, num_sms=152, l2_bytes=L2)[0] == 0
    assert bd.attn_a2a_split_plan(1, 24, 4608, 128, split=bd.SPLIT_ALL, num_sms=152, l2_bytes=L2) == (bd.SPLIT_ALL, 0, 103)
    assert bd.attn_a2a_split_plan(1, 40, 32768, 128, num_sms=152, l2_bytes=L2) == (bd.SPLIT_TAIL, 5016, 176)
    assert bd.attn_a2a_split_plan(1, 40, 4096, 128, num_sms=152, l2_bytes=L2)[0] == 0
    assert bd.attn_a2a_split_plan(1, 24, 4096, 128, split=bd.SPLIT_NONE, num_sms=152, l2_bytes=L2)[0] == 0
    # a grid larger than the SM count is never split (its CTAs need not all be resident)
    assert bd.attn_a2a_split_plan(1, 24, 4096, 128, grid=200, num_sms=152, l2_bytes=L2)[0] == 0
    out = [ctypes.c_int(0) for _ in range(3)]
    ptrs = [ctypes.byref(x) for x in out]
    for args in ((1, 24, 4096, 96, 0, 152, L2, 0), (1, 24, 4096, 128, -1, 152, L2, 0),
                 (1, 24, 4096, 128, 0, 152, L2, 4), (-1, 24, 4096, 128, 0, 152, L2, 0)):
        assert lib.attn_a2a_split_plan(*args, *ptrs) == bd.EINVAL
    assert lib.attn_a2a_split_plan(1, 24, 4096, 128, 0, 152, L2, 0, None, ptrs[1], ptrs[2]) == bd.EINVAL


def test_empty_problem_is_ok_without_launch(lib):
    # S = 0: every chunk is empty, null partitions are allowed, nothing is launched
    assert call_fwd(lib, S=0, parts=[0, 0]) == bd.OK
    assert call_fwd(lib, B=0, parts=[0, 0]) == bd.OK


def test_contig_and_permute_validation(lib):
    shp = bd.plain_shape(1, 4, 256, 64)
    assert lib.attn_a2a_fwd_contig_ex(FAKE, FAKE * 2, FAKE * 3, ctypes.byref(shp), 0.1, FAKE * 16, None,
                                      ctypes.byref(bd._opts(store_kind=4)), None) == bd.EINVAL
    # whole-line row stores are built for the all-to-all layout only (refused before any launch)
    assert lib.attn_a2a_fwd_contig_ex(FAKE, FAKE * 2, FAKE * 3, ctypes.byref(shp), 0.1, FAKE * 16, None,
                                      ctypes.byref(bd._opts(store_kind=3)), None) == bd.EUNSUPPORTED
    assert lib.attn_a2a_fwd_contig(FAKE, FAKE * 2, FAKE * 3, ctypes.byref(shp), 0.1, None, None, None) == bd.EINVAL
    # output overlapping q
    assert lib.attn_a2a_fwd_contig(FAKE, FAKE * 4, FAKE * 8, ctypes.byref(shp), 0.1, FAKE + 64, None, None) == bd.EINVAL
    parts = (ctypes.c_void_p * 2)(FAKE * 16, FAKE * 17)
    assert lib.attn_a2a_permute(None, ctypes.byref(shp), 2, parts, None) == bd.EINVAL
    assert lib.attn_a2a_permute(FAKE, ctypes.byref(shp), 3, parts, None) == bd.EINVAL
    bad = bd.plain_shape(1, 4, 256, 80)
    assert lib.attn_a2a_permute(FAKE, ctypes.byref(bad), 2, parts, None) == bd.EUNSUPPORTED


def test_probe_validation(lib):
    def run(**kw):
        c = dict(K=4, rounds=3, V_bytes=4096 * 4, G_ns=0, store_kind=0, gap_kind=0, dst=FAKE,
                 dst_bytes=4096 * 16, stamps=FAKE, fma_iters=0)
        c.update(kw)
        cfg = bd.ProbeCfg(c["K"], c["rounds"], c["V_bytes"], c["G_ns"], c["store_kind"], c["gap_kind"],
                          c["dst"], c["dst_bytes"], c["stamps"], c["fma_iters"])
        return lib.xstage_probe_run(ctypes.byref(cfg), None)

    assert run(K=0) == bd.EINVAL
    assert run(rounds=0) == bd.EINVAL
    assert run(V_bytes=4096 * 4 + 16) == bd.EINVAL
    assert run(dst_bytes=4096) == bd.EINVAL
    assert run(store_kind=3) == bd.EINVAL
    assert run(G_ns=-1) == bd.EINVAL
    assert run(stamps=0) == bd.EINVAL
    assert run(dst=FAKE + 4) == bd.EINVAL


def test_chunk_sizes_rule():
    assert bd.chunk_sizes(75600, 8) == [9450] * 8
    assert bd.chunk_sizes(10, 4) == [3, 3, 2, 2]
    assert bd.chunk_sizes(3, 8) == [1, 1, 1, 0, 0, 0, 0, 0]


def test_noalloc_probe_validation(lib):
    def run(**kw):
        c = dict(K=4, rounds=3, V_bytes=4096 * 4, G_ns=0, store_kind=0, gap_kind=0, stamps=FAKE, fma_iters=0)
        c.update(kw)
        cfg = bd.ProbeCfg(c["K"], c["rounds"], c["V_bytes"], c["G_ns"], c["store_kind"], c["gap_kind"],
                          None, 0, c["stamps"], c["fma_iters"])
        return lib.xstage_probe_run_noalloc(ctypes.byref(cfg), None)

    assert run(V_bytes=bd.NOALLOC_MAX_BYTES + 4096 * 4) == bd.ETOOLARGE
    assert run(K=0) == bd.EINVAL
    assert run(stamps=0) == bd.EINVAL
    assert run(store_kind=3) == bd.EINVAL
    assert run(gap_kind=1, fma_iters=10**8 + 1) == bd.EINVAL
    assert run(gap_kind=2, fma_iters=10**8 + 1) == bd.EINVAL
    assert "scratch" in bd.strerror(bd.ETOOLARGE)


# Invalid probe configurations: both probe entry points must return the same
# status for each (they share their field checks; only the burst target differs).
BAD_PROBE_FIELDS = [
    dict(K=0), dict(K=1025), dict(rounds=0), dict(V_bytes=0), dict(V_bytes=4096 * 4 + 16),
    dict(G_ns=-1), dict(store_kind=-1), dict(store_kind=3), dict(gap_kind=-1), dict(gap_kind=3),
    dict(gap_kind=1, fma_iters=-1), dict(gap_kind=1, fma_iters=10**8 + 1),
    dict(gap_kind=2, fma_iters=-1), dict(gap_kind=2, fma_iters=10**8 + 1),
    dict(stamps=0), dict(stamps=FAKE + 4),
]


@pytest.mark.parametrize("bad", BAD_PROBE_FIELDS, ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_probe_entry_points_validate_alike(lib, bad):
    c = dict(K=4, rounds=3, V_bytes=4096 * 4, G_ns=0, store_kind=0, gap_kind=0, stamps=FAKE, fma_iters=0)
    c.update(bad)

    def cfg(dst, dst_bytes):
        return bd.ProbeCfg(c["K"], c["rounds"], c["V_bytes"], c["G_ns"], c["store_kind"], c["gap_kind"],
                           dst, dst_bytes, c["stamps"], c["fma_iters"])

    rc_run = lib.xstage_probe_run(ctypes.byref(cfg(FAKE, 4096 * 64)), None)
    rc_noalloc = lib.xstage_probe_run_noalloc(ctypes.byref(cfg(None, 0)), None)
    assert rc_run == bd.EINVAL
    assert rc_noalloc == rc_run


def test_s2s_validation(lib):
    shp = bd.plain_shape(1, 16, 256, 64)
    ptrs = lambda base, n: (ctypes.c_void_p * n)(*[FAKE * (base + j) for j in range(n)])
    # P beyond the 8 tensor maps the kernel carries
    assert lib.attn_a2a_fwd_s2s(ptrs(100, 16), ptrs(200, 16), ptrs(300, 16), ctypes.byref(shp), 16, 0.1,
                                ptrs(400, 16), None, None) == bd.EUNSUPPORTED
    # null input partition
    q = ptrs(100, 2)
    q[1] = None
    assert lib.attn_a2a_fwd_s2s(q, ptrs(200, 2), ptrs(300, 2), ctypes.byref(shp), 2, 0.1, ptrs(400, 2),
                                None, None) == bd.EINVAL
    # output partition aliasing an input partition
    assert lib.attn_a2a_fwd_s2s(ptrs(100, 2), ptrs(200, 2), ptrs(300, 2), ctypes.byref(shp), 2, 0.1,
                                ptrs(200, 2), None, None) == bd.EINVAL
    assert lib.attn_a2a_fwd_s2s(None, ptrs(200, 2), ptrs(300, 2), ctypes.byref(shp), 2, 0.1, ptrs(400, 2),
                                None, None) == bd.EINVAL


def test_moe_validation(lib):
    dst = (ctypes.c_void_p * 2)(FAKE * 20, FAKE * 21)
    rows = (ctypes.c_int * 2)(64, 64)

    def run(E=2, T=128, K=128, N=256, n_tasks=4, P=2):
        return lib.moe_gemm_scatter(FAKE, FAKE * 2, FAKE * 3, E, T, K, N, FAKE * 4, n_tasks, FAKE * 5,
                                    FAKE * 6, P, dst, rows, None, 0, None)

    assert run(N=128) == bd.EINVAL  # a task is 256 output columns wide
    assert run(N=384) == bd.EINVAL
    assert run(T=100) == bd.EINVAL
    assert run(K=96) == bd.EINVAL
    assert run(P=0) == bd.EINVAL
    assert run(n_tasks=-1) == bd.EINVAL
    assert run(n_tasks=0) == bd.OK  # nothing to do, nothing launched


def test_part_heads_validation(lib):
    def run(H=4, P=2, part_heads=0, a2a=True):
        opts = bd._opts(part_heads=part_heads)
        shp = bd.plain_shape(1, H, 256, 64)
        parts = (ctypes.c_void_p * P)(*[FAKE * (16 + j) for j in range(P)])
        if a2a:
            return lib.attn_a2a_fwd_ex(FAKE, FAKE * 2, FAKE * 3, ctypes.byref(shp), P, 0.125, parts, None,
                                       ctypes.byref(opts), None)
        return lib.attn_a2a_fwd_contig_ex(FAKE, FAKE * 2, FAKE * 3, ctypes.byref(shp), 0.125, FAKE * 16, None,
                                          ctypes.byref(opts), None)

    assert run(H=4, part_heads=2) == bd.EINVAL          # fewer heads per row than the call computes
    assert run(H=2, P=4, part_heads=6) == bd.EINVAL     # a row of 6 heads does not split over 4 ranks
    assert run(H=1, P=4, part_heads=4, a2a=False) == bd.EINVAL  # contiguous layout has no partitions
    assert run(part_heads=-1) == bd.EINVAL

