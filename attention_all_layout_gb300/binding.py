"""Thin ctypes binding of libattn_a2a.so (include/attn_a2a.h).

Argument marshalling only: tensors become raw pointers, shapes and strides
become the C structs, the current torch CUDA stream becomes the cudaStream_t.
Every step of the computation runs in the library's CUDA kernels. There is
no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_a2a.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, ETIMEOUT, ETOOLARGE = 0, 1, 2, 3, 4, 5
MAX_RANKS = 64
NOALLOC_MAX_BYTES = 16 * 1024 * 1024  # XSTAGE_PROBE_NOALLOC_MAX_BYTES

# Every symbol include/attn_a2a.h declares.
EXPORTED = (
    "attn_a2a_fwd",
    "attn_a2a_fwd_ex",
    "attn_a2a_fwd_contig",
    "attn_a2a_fwd_contig_ex",
    "attn_a2a_fwd_s2s",
    "attn_a2a_fwd_s2s_ex",
    "attn_a2a_permute",
    "attn_a2a_fwd_simt",
    "attn_a2a_fwd_host",
    "xstage_probe_run",
    "xstage_probe_run_noalloc",
    "moe_gemm_scatter",
    "attn_a2a_strerror",
    "attn_a2a_num_sms",
    "attn_a2a_store_kind",
    "attn_a2a_split_plan",
)


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("S", ctypes.c_int), ("d", ctypes.c_int)] + [
        (n, ctypes.c_longlong)
        for n in ("q_sb", "q_sh", "q_ss", "k_sb", "k_sh", "k_ss", "v_sb", "v_sh", "v_ss")
    ]


class Opts(ctypes.Structure):
    _fields_ = [
        ("store_kind", ctypes.c_int),
        ("grid", ctypes.c_int),
        ("timeout_ns", ctypes.c_longlong),
        ("inject_stall", ctypes.c_int),
        ("tile_order", ctypes.c_int),
        ("trace", ctypes.c_void_p),
        ("part_heads", ctypes.c_int),
        ("split", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_longlong),
        ("cta_pairs", ctypes.c_int),
    ]


class ProbeCfg(ctypes.Structure):
    _fields_ = [
        ("K", ctypes.c_int),
        ("rounds", ctypes.c_int),
        ("V_bytes", ctypes.c_longlong),
        ("G_ns", ctypes.c_longlong),
        ("store_kind", ctypes.c_int),
        ("gap_kind", ctypes.c_int),
        ("dst", ctypes.c_void_p),
        ("dst_bytes", ctypes.c_longlong),
        ("stamps", ctypes.c_void_p),
        ("fma_iters", ctypes.c_longlong),
    ]


class AttnA2AError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (status {code})")
        self.code = code


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m attention_all_layout_gb300.build` "
            "(there is no CPU or PyTorch fallback)"
        )
    lib = ctypes.CDLL(path)
    vp, cint = ctypes.c_void_p, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    shp = ctypes.POINTER(Shape)
    opt = ctypes.POINTER(Opts)
    lib.attn_a2a_fwd.argtypes = [vp, vp, vp, shp, cint, ctypes.c_float, pp, vp, vp]
    lib.attn_a2a_fwd_ex.argtypes = [vp, vp, vp, shp, cint, ctypes.c_float, pp, vp, opt, vp]
    lib.attn_a2a_fwd_contig.argtypes = [vp, vp, vp, shp, ctypes.c_float, vp, vp, vp]
    lib.attn_a2a_fwd_contig_ex.argtypes = [vp, vp, vp, shp, ctypes.c_float, vp, vp, opt, vp]
    lib.attn_a2a_fwd_s2s.argtypes = [pp, pp, pp, shp, cint, ctypes.c_float, pp, vp, vp]
    lib.attn_a2a_fwd_s2s_ex.argtypes = [pp, pp, pp, shp, cint, ctypes.c_float, pp, vp, ctypes.POINTER(Opts), vp]
    lib.attn_a2a_permute.argtypes = [vp, shp, cint, pp, vp]
    lib.attn_a2a_fwd_simt.argtypes = [vp, vp, vp, shp, cint, ctypes.c_float, pp, vp]
    lib.attn_a2a_fwd_host.argtypes = [vp, vp, vp, shp, cint, ctypes.c_float, vp, vp, vp, pp, pp, vp, vp]
    lib.xstage_probe_run.argtypes = [ctypes.POINTER(ProbeCfg), vp]
    lib.xstage_probe_run_noalloc.argtypes = [ctypes.POINTER(ProbeCfg), vp]
    lib.moe_gemm_scatter.argtypes = [vp, vp, vp, cint, cint, cint, cint, vp, cint, vp, vp, cint, pp,
                                     ctypes.POINTER(ctypes.c_int), vp, cint, vp]
    lib.attn_a2a_strerror.argtypes = [cint]
    lib.attn_a2a_strerror.restype = ctypes.c_char_p
    lib.attn_a2a_num_sms.argtypes = []
    lib.attn_a2a_store_kind.argtypes = [cint, cint, cint, cint, ctypes.POINTER(ctypes.c_int)]
    ip = ctypes.POINTER(ctypes.c_int)
    lib.attn_a2a_split_plan.argtypes = [cint, cint, cint, cint, cint, cint, ctypes.c_longlong, cint, ip, ip, ip]
    for name in EXPORTED:
        if name != "attn_a2a_strerror":
            getattr(lib, name).restype = cint
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().attn_a2a_strerror(int(code)).decode()


def num_sms() -> int:
    return int(load().attn_a2a_num_sms())


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def shape_of(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> Shape:
    """attn_a2a_shape of [B, H, S, d] tensors (innermost stride must be 1)."""
    B, H, S, d = q.shape
    for t in (q, k, v):
        if t.dim() != 4 or tuple(t.shape) != (B, H, S, d):
            raise ValueError("q, k, v must share one [B, H, S, d] shape")
        if t.dtype != torch.bfloat16:
            raise ValueError("q, k, v must be bf16")
        if d > 0 and t.stride(3) != 1 and t.numel() > 0:
            raise ValueError("the head dimension must be contiguous")
    return Shape(B, H, S, d, *q.stride()[:3], *k.stride()[:3], *v.stride()[:3])


def plain_shape(B: int, H: int, S: int, d: int) -> Shape:
    sb, sh, ss = H * S * d, S * d, d
    return Shape(B, H, S, d, sb, sh, ss, sb, sh, ss, sb, sh, ss)


def chunk_sizes(S: int, P: int) -> list[int]:
    """Rows of each of the P sequence chunks (larger chunks first)."""
    base, rem = divmod(S, P)
    return [base + (1 if j < rem else 0) for j in range(P)]


def alloc_partitions(B: int, S: int, H: int, d: int, P: int, device="cuda", fill=None):
    """P contiguous bf16 partitions [B, c_j, H, d] on `device`."""
    parts = []
    for c in chunk_sizes(S, P):
        t = torch.empty((B, c, H, d), dtype=torch.bfloat16, device=device)
        if fill is not None:
            t.fill_(fill)
        parts.append(t)
    return parts


def _ptr_array(tensors: Sequence):
    """Host array of device pointers: tensors (empty ones as NULL), raw integer
    addresses (e.g. offsets into partitions shared by several head groups), or None."""
    arr = (ctypes.c_void_p * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        if isinstance(t, int):
            arr[i] = t or None
        else:
            arr[i] = None if (t is None or t.numel() == 0) else t.data_ptr()
    return arr


SPLIT_AUTO, SPLIT_TAIL, SPLIT_ALL, SPLIT_NONE = 0, 1, 2, 3  # attn_a2a_opts.split
PAIRS_AUTO, PAIRS_ON, PAIRS_OFF = 0, 1, 2  # attn_a2a_opts.cta_pairs


def _opts(store_kind=0, grid=0, timeout_ns=0, inject_stall=0, tile_order=0, trace=None, part_heads=0,
          workspace=None, split=SPLIT_AUTO, cta_pairs=PAIRS_AUTO) -> Opts:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return Opts(store_kind, grid, timeout_ns, inject_stall, tile_order, _ptr(trace), part_heads, split,
                _ptr(workspace), ws_bytes, cta_pairs)


def workspace_bytes(grid: int, d: int) -> int:
    """Bytes of the split-tail workspace for `grid` CTAs and head dim d (the header's
    ATTN_A2A_WORKSPACE_BYTES)."""
    return 256 + 32 * grid + 1024 * grid * (d + 2)


def alloc_workspace(d: int = 128, grid: int = 0, device="cuda") -> torch.Tensor:
    """A zeroed split-tail workspace (attn_a2a_opts.workspace) for up to `grid` CTAs
    (0 = one per SM). Reusable by every later call on the same stream."""
    g = grid or num_sms()
    return torch.zeros(workspace_bytes(g, d), dtype=torch.uint8, device=device)


TRACE_RECORD = 8  # int64 per (work item, query tile, warp) of a traced call


def trace_numel(B: int, H: int, S: int) -> int:
    """int64 elements of the trace buffer of a traced call (the header's ATTN_A2A_TRACE_BYTES / 8)."""
    pairs = ((S + 127) // 128 + 1) // 2
    return B * H * pairs * 2 * 4 * TRACE_RECORD


def _check_trace(trace, shp) -> None:
    if trace is None:
        return
    if trace.dtype != torch.int64 or not trace.is_cuda or not trace.is_contiguous():
        raise ValueError("trace must be a contiguous int64 CUDA tensor")
    if trace.numel() < trace_numel(shp.B, shp.H, shp.S):
        raise ValueError(f"trace needs {trace_numel(shp.B, shp.H, shp.S)} int64 elements")


def _check(code: int, what: str, check: bool) -> int:
    if check and code != OK:
        raise AttnA2AError(code, what)
    return code


# ------------------------------------------------------------------ entry points (same names as the C ABI)
def attn_a2a_fwd(q, k, v, P: int, scale: float, out_partitions, dev_status=None, stream=None,
                 store_kind: int = 0, grid: int = 0, timeout_ns: int = 0, inject_stall: int = 0,
                 tile_order: int = 0, trace=None, part_heads: int = 0, workspace=None, split: int = SPLIT_AUTO,
                 cta_pairs: int = PAIRS_AUTO, check: bool = True) -> int:
    """Fused attention + head->sequence all-to-all into `out_partitions` (P tensors [B,c_j,H,d]).
    trace: optional device int64 tensor of trace_numel(B, H, S) elements for per-tile stamps.
    part_heads: heads per partition row for a head-group launch (0 = H); the partitions are then
    given as device addresses already offset to the group's first head (see ulysses.py).
    workspace: optional zeroed uint8 tensor (alloc_workspace) that lets work items be split over
    all CTAs by key blocks; split: which (SPLIT_AUTO, SPLIT_TAIL, SPLIT_ALL, SPLIT_NONE).
    cta_pairs: PAIRS_ON runs the work on two-CTA clusters sharing each K/V block (M = 256 MMAs),
    PAIRS_OFF one CTA per item, PAIRS_AUTO lets the library choose."""
    lib = load()
    shp = shape_of(q, k, v)
    parts = _ptr_array(out_partitions)
    _check_trace(trace, shp)
    opts = _opts(store_kind, grid, timeout_ns, inject_stall, tile_order, trace, part_heads, workspace, split,
                 cta_pairs)
    rc = lib.attn_a2a_fwd_ex(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(shp), int(P), float(scale), parts,
                             _ptr(dev_status), ctypes.byref(opts), _stream(stream))
    return _check(rc, "attn_a2a_fwd", check)


def attn_a2a_fwd_contig(q, k, v, scale: float, out, dev_status=None, stream=None, store_kind: int = 0,
                        grid: int = 0, timeout_ns: int = 0, trace=None, workspace=None, split: int = SPLIT_AUTO,
                        cta_pairs: int = PAIRS_AUTO, check: bool = True) -> int:
    """The same kernel with a contiguous [B, H, S, d] output ("attention alone")."""
    lib = load()
    shp = shape_of(q, k, v)
    _check_trace(trace, shp)
    opts = _opts(store_kind, grid, timeout_ns, 0, 0, trace, 0, workspace, split, cta_pairs)
    rc = lib.attn_a2a_fwd_contig_ex(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(shp), float(scale), _ptr(out),
                                    _ptr(dev_status), ctypes.byref(opts), _stream(stream))
    return _check(rc, "attn_a2a_fwd_contig", check)


def attn_a2a_fwd_s2s(q_parts, k_parts, v_parts, P: int, scale: float, out_partitions, dev_status=None,
                     stream=None, store_kind: int = 0, grid: int = 0, timeout_ns: int = 0, workspace=None,
                     split: int = SPLIT_AUTO, check: bool = True) -> int:
    """Sequence-sharded q, k, v partitions [B, c_j, H, d] in, sequence-sharded output out.
    workspace / split: the split schedule, as for attn_a2a_fwd (where tiles are counted over
    the whole sequence)."""
    lib = load()
    B, _, H, d = q_parts[0].shape
    S = sum(t.shape[1] for t in q_parts)
    for parts in (q_parts, k_parts, v_parts):
        for t in parts:
            if t.dtype != torch.bfloat16 or (t.numel() and not t.is_contiguous()):
                raise ValueError("partitions must be contiguous bf16 [B, c_j, H, d]")
    shp = plain_shape(B, H, S, d)
    opts = _opts(store_kind, grid, timeout_ns, 0, 0, None, 0, workspace, split)
    rc = lib.attn_a2a_fwd_s2s_ex(_ptr_array(q_parts), _ptr_array(k_parts), _ptr_array(v_parts), ctypes.byref(shp),
                                 int(P), float(scale), _ptr_array(out_partitions), _ptr(dev_status),
                                 ctypes.byref(opts), _stream(stream))
    return _check(rc, "attn_a2a_fwd_s2s", check)


def attn_a2a_permute(o, P: int, out_partitions, stream=None, check: bool = True) -> int:
    """Separate all-to-all copy of a contiguous [B, H, S, d] tensor into the partitions."""
    lib = load()
    B, H, S, d = o.shape
    shp = plain_shape(B, H, S, d)
    rc = lib.attn_a2a_permute(_ptr(o), ctypes.byref(shp), int(P), _ptr_array(out_partitions), _stream(stream))
    return _check(rc, "attn_a2a_permute", check)


def attn_a2a_fwd_simt(q, k, v, P: int, scale: float, out_partitions, stream=None, check: bool = True) -> int:
    """Slow SIMT debug path with the same partition epilogue."""
    lib = load()
    shp = shape_of(q, k, v)
    rc = lib.attn_a2a_fwd_simt(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(shp), int(P), float(scale),
                               _ptr_array(out_partitions), _stream(stream))
    return _check(rc, "attn_a2a_fwd_simt", check)


def attn_a2a_fwd_host(hq, hk, hv, P: int, scale: float, dq, dk, dv, dparts, hparts, dev_status=None,
                      stream=None, check: bool = True) -> int:
    """Host-memory variant: H2D copies, fused kernel, D2H copies, all enqueued on `stream`."""
    lib = load()
    B, H, S, d = hq.shape
    shp = plain_shape(B, H, S, d)
    rc = lib.attn_a2a_fwd_host(_ptr(hq), _ptr(hk), _ptr(hv), ctypes.byref(shp), int(P), float(scale),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr_array(dparts), _ptr_array(hparts),
                               _ptr(dev_status), _stream(stream))
    return _check(rc, "attn_a2a_fwd_host", check)


def xstage_probe_run(K: int, rounds: int, V_bytes: int, G_ns: int, dst: torch.Tensor, stamps: torch.Tensor,
                     store_kind: int = 0, gap_kind: int = 0, fma_iters: int = 0, stream=None,
                     check: bool = True) -> int:
    """One Burst-Gap probe launch; per-round stamps land in `stamps` (int64 [K, rounds, 3])."""
    lib = load()
    cfg = ProbeCfg(int(K), int(rounds), int(V_bytes), int(G_ns), int(store_kind), int(gap_kind),
                   _ptr(dst), dst.numel() * dst.element_size(), _ptr(stamps), int(fma_iters))
    rc = lib.xstage_probe_run(ctypes.byref(cfg), _stream(stream))
    return _check(rc, "xstage_probe_run", check)


def xstage_probe_run_noalloc(K: int, rounds: int, V_bytes: int, G_ns: int, stamps: torch.Tensor,
                             store_kind: int = 0, gap_kind: int = 0, fma_iters: int = 0, stream=None,
                             check: bool = True) -> int:
    """The probe for callers that cannot allocate: the burst target is the library's fixed
    16 MiB device array (no dst argument); per-round stamps land in `stamps`."""
    lib = load()
    cfg = ProbeCfg(int(K), int(rounds), int(V_bytes), int(G_ns), int(store_kind), int(gap_kind),
                   None, 0, _ptr(stamps), int(fma_iters))
    rc = lib.xstage_probe_run_noalloc(ctypes.byref(cfg), _stream(stream))
    return _check(rc, "xstage_probe_run_noalloc", check)


def moe_gemm_scatter(x, w1, w2, tasks, h_out, row_map, dst, dev_status=None, grid: int = 0, stream=None,
                     check: bool = True) -> int:
    """Grouped GEMM task list (kind 0: h_out tile; kind 1: scattered rows into dst[rank])."""
    lib = load()
    E, T, K = x.shape
    N = w1.shape[1]
    for t in (x, w1, w2, h_out):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("x, w1, w2, h_out must be contiguous bf16")
    if tasks.dtype != torch.int32 or row_map.dtype != torch.int32:
        raise ValueError("tasks and row_map must be int32")
    rows = (ctypes.c_int * len(dst))(*[int(d.shape[0]) for d in dst])
    rc = lib.moe_gemm_scatter(_ptr(x), _ptr(w1), _ptr(w2), E, T, K, N, _ptr(tasks), int(tasks.shape[0]), _ptr(h_out),
                              _ptr(row_map), len(dst), _ptr_array(dst), rows, _ptr(dev_status), int(grid),
                              _stream(stream))
    return _check(rc, "moe_gemm_scatter", check)


def attn_a2a_strerror(code: int) -> str:
    return strerror(code)


def attn_a2a_num_sms() -> int:
    return num_sms()


def attn_a2a_split_plan(B: int, H: int, S: int, d: int, grid: int = 0, split: int = SPLIT_AUTO, num_sms: int = 0,
                        l2_bytes: int = 0):
    """The split schedule a call with a workspace would use: (kind, first item, key blocks per
    CTA range); kind SPLIT_ALL, SPLIT_TAIL or 0. num_sms / l2_bytes 0 = the current device's."""
    kind, first, blocks = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = load().attn_a2a_split_plan(int(B), int(H), int(S), int(d), int(grid), int(num_sms), int(l2_bytes),
                                    int(split), ctypes.byref(kind), ctypes.byref(first), ctypes.byref(blocks))
    _check(rc, "attn_a2a_split_plan", True)
    return kind.value, first.value, blocks.value


def attn_a2a_store_kind(S: int, P: int, layout: int, store_kind: int = 0) -> int:
    """Store kind the library uses for these sizes: 1 = bulk tensor stores, 2 = row stores,
    3 = whole-line row stores (all-to-all layout, on request only).
    layout 0 = contiguous (attention alone), 1 = all-to-all. Raises AttnA2AError on a bad request."""
    out = ctypes.c_int(0)
    rc = load().attn_a2a_store_kind(int(S), int(P), int(layout), int(store_kind), ctypes.byref(out))
    _check(rc, "attn_a2a_store_kind", True)
    return out.value
