"""CPU oracle for MoE token layout -> dispatch -> combine (numpy front end).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
library never imports, links or executes anything here, and this package
imports nothing from the product package: the two share no code.  The only
shared module is the seeded input generator, which holds none of the method's
arithmetic.

The arithmetic lives in ``ep_oracle.c`` (plain single-threaded C, one loop per
step, each function citing the passage it follows).  This module only
marshals numpy arrays, except for the SM count rule, a few lines of host
arithmetic written here in Python with exact binomial coefficients.

Pins (CPU tests): an independent numpy filter-and-sort formulation of the
layout on small inputs; the count invariants of "DeepEP Symmetric Memory"
section 7.3; the expected-distinct-groups closed form of the
``get_theoretical_num_sms`` fragment of "DeepEP V2 ElasticBuffer architecture";
the exact dispatch -> identity -> combine closed form; the OCP E4M3 definition
and torch's CPU float8 cast.
"""
import ctypes
import math

import numpy as np

from . import build as _build

_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


_lib_omp = None


class threads:
    """``with oracle.threads() as n:`` -- the calls inside run on the OpenMP
    build of the same C source (token loops of dispatch and combine split
    over ``n`` host threads; the layout stays sequential).  n is None, and
    the single-threaded build stays in use, when no OpenMP build exists.
    For the benchmark's all-cores CPU baseline."""

    def __enter__(self):
        global _lib, _lib_omp
        self._saved = _load()
        if _lib_omp is None:
            path = _build.build_omp()
            if path is None:
                return None
            _lib_omp = _configure(ctypes.CDLL(path))
        _lib = _lib_omp
        return int(_lib_omp.ep_oracle_threads())

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _configure(lib):
    vp = ctypes.c_void_p
    lib.ep_oracle_threads.restype = ctypes.c_int
    lib.ep_oracle_threads.argtypes = []
    lib.ep_oracle_layout.restype = ctypes.c_int
    lib.ep_oracle_layout.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int] + [vp] * 11
    lib.ep_oracle_dispatch.restype = ctypes.c_int
    lib.ep_oracle_dispatch.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int64, vp, vp, vp, vp, vp, vp]
    lib.ep_oracle_combine.restype = ctypes.c_int
    lib.ep_oracle_combine.argtypes = [vp, ctypes.c_int64, vp, vp, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      vp, vp, ctypes.c_int, vp]
    lib.ep_oracle_fp8_cast_row.restype = None
    lib.ep_oracle_fp8_cast_row.argtypes = [vp, ctypes.c_int, vp, vp]
    lib.ep_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.ep_oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.ep_oracle_e4m3_decode.restype = ctypes.c_float
    lib.ep_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.ep_oracle_float_to_bf16.restype = ctypes.c_uint16
    lib.ep_oracle_float_to_bf16.argtypes = [ctypes.c_float]
    lib.ep_oracle_bf16_to_float.restype = ctypes.c_float
    lib.ep_oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
    lib.ep_oracle_expanded_rows.restype = ctypes.c_int
    lib.ep_oracle_expanded_rows.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    lib.ep_oracle_dispatch_expanded.restype = ctypes.c_int
    lib.ep_oracle_dispatch_expanded.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp,
                                                ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                vp, vp, vp, vp]
    lib.ep_oracle_combine_expanded.restype = ctypes.c_int
    lib.ep_oracle_combine_expanded.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, vp, vp]
    lib.ep_oracle_combine_topk_weights.restype = ctypes.c_int
    lib.ep_oracle_combine_topk_weights.argtypes = [vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, vp, vp]
    lib.ep_oracle_accumulate_expert_stats.restype = None
    lib.ep_oracle_accumulate_expert_stats.argtypes = [vp, ctypes.c_int, vp]
    for name in ("ep_oracle_e4m3_encode_array", "ep_oracle_e4m3_decode_array",
                 "ep_oracle_float_to_bf16_array"):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [vp, ctypes.c_int64, vp]
    lib.ep_oracle_double_to_bf16_array.restype = None
    lib.ep_oracle_double_to_bf16_array.argtypes = [vp, ctypes.c_int64, vp]
    lib.ep_oracle_node_rows.restype = ctypes.c_int
    lib.ep_oracle_node_rows.argtypes = [vp] + [ctypes.c_int] * 5 + [vp, vp]
    lib.ep_oracle_dispatch_hierarchical.restype = ctypes.c_int
    lib.ep_oracle_dispatch_hierarchical.argtypes = (
        [vp, vp, vp] + [ctypes.c_int] * 6 + [vp, vp, ctypes.c_int, ctypes.c_int64, vp, vp, vp, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int64, vp, vp, vp, vp, vp])
    lib.ep_oracle_combine_hierarchical.restype = ctypes.c_int
    lib.ep_oracle_combine_hierarchical.argtypes = (
        [vp, ctypes.c_int64, vp, vp] + [ctypes.c_int] * 7 + [vp, vp, ctypes.c_int64, vp, vp, vp])
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


EP_ERR_INVALID_INDEX = 4
EP_ERR_CAPACITY = 8


class Layout:
    """Result of :func:`layout` (all numpy int32 / uint8 arrays)."""

    def __init__(self, **kw):
        self.__dict__.update(kw)

    @property
    def num_recv(self):
        return int(self.rank_offset[-1])


def layout(topk_idx, E, R, ranks_per_node=0, expert_alignment=1, with_src_dst=True):
    """Routing layout of int64 ``topk_idx`` [T, K] (see ep_oracle_layout)."""
    lib = _load()
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    nodes = R // ranks_per_node if ranks_per_node > 0 else 0
    out = Layout(
        num_tokens_per_rank=np.zeros(R, np.int32),
        num_tokens_per_node=np.zeros(nodes, np.int32) if nodes else None,
        num_tokens_per_expert=np.zeros(E, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        rank_offset=np.zeros(R + 1, np.int32),
        expert_offset=np.zeros(E + 1, np.int32),
        dst_row=np.zeros((T, R), np.int32),
        src_dst_count=np.zeros((R, R), np.int32) if (with_src_dst and T % R == 0) else None,
        token_offset=np.zeros(T + 1, np.int32),
    )
    scratch_local = np.zeros(max(T * R, 1), np.int32)
    scratch_mark = np.zeros(R + max(nodes, 1), np.uint8)
    status = lib.ep_oracle_layout(
        _p(topk_idx), T, K, E, R, ranks_per_node, expert_alignment,
        _p(out.num_tokens_per_rank), _p(out.num_tokens_per_node), _p(out.num_tokens_per_expert),
        _p(out.is_token_in_rank), _p(out.rank_offset), _p(out.expert_offset), _p(out.dst_row),
        _p(out.src_dst_count), _p(out.token_offset), _p(scratch_local), _p(scratch_mark))
    out.status = status
    return out


def dispatch(x_bits, topk_idx, topk_weights, E, R, dst_row, capacity=None, fp8=False,
             sf_col_major=False, sf_stride=None, tokens=None):
    """Dispatch (see ep_oracle_dispatch).

    ``x_bits``: uint16 [T, H] bf16 bit patterns.  With ``tokens`` given, the
    result is compact: rows numbered in (listed token, rank) order and the
    returned dict carries ``rows`` (each row's destination index).
    """
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    dst_row = np.ascontiguousarray(dst_row, dtype=np.int32)
    T, H = x_bits.shape
    K = topk_idx.shape[1]
    compact = tokens is not None
    if compact:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        n_rows = int((dst_row[tokens] >= 0).sum())
    else:
        n_rows = int(capacity if capacity is not None else (dst_row.max() + 1 if dst_row.size else 0))
    n_alloc = max(n_rows, 1)
    row_bytes = H if fp8 else 2 * H
    nb = H // 128
    if sf_stride is None:
        sf_stride = n_alloc
    recv_x = np.zeros((n_alloc, row_bytes), np.uint8)
    recv_sf = None
    if fp8:
        recv_sf = np.zeros(nb * sf_stride if sf_col_major else n_alloc * nb, np.float32)
    recv_topk_idx = np.zeros((n_alloc, K), np.int32)
    recv_topk_weights = np.zeros((n_alloc, K), np.float32)
    recv_src_idx = np.zeros(n_alloc, np.int32)
    rows = np.zeros(n_alloc, np.int32) if compact else None
    status = lib.ep_oracle_dispatch(
        _p(x_bits), _p(topk_idx), _p(topk_weights), T, H, K, E, R, _p(dst_row),
        _p(tokens), len(tokens) if compact else 0, 1 if compact else 0, n_rows,
        1 if fp8 else 0, 1 if sf_col_major else 0, sf_stride,
        _p(recv_x), _p(recv_sf), _p(recv_topk_idx), _p(recv_topk_weights), _p(recv_src_idx),
        _p(rows))
    res = dict(recv_x=recv_x[:n_rows], recv_topk_idx=recv_topk_idx[:n_rows],
               recv_topk_weights=recv_topk_weights[:n_rows], recv_src_idx=recv_src_idx[:n_rows],
               status=status)
    if fp8:
        res["recv_sf"] = recv_sf if sf_col_major else recv_sf.reshape(n_alloc, nb)[:n_rows]
    if compact:
        res["rows"] = rows[:n_rows]
    return res


def combine(y_bits, topk_idx, topk_weights, E, R, dst_row, weighted=False, tokens=None):
    """Combine (see ep_oracle_combine); returns float64 [len(tokens) or T, H]."""
    lib = _load()
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    H = y_bits.shape[1]
    if topk_weights is None:
        topk_weights = np.zeros((T, K), np.float32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    dst_row = np.ascontiguousarray(dst_row, dtype=np.int32)
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        n = len(tokens)
    else:
        n = T
    out = np.zeros((max(n, 1), H), np.float64)
    status = lib.ep_oracle_combine(_p(y_bits), y_bits.shape[0], _p(topk_idx), _p(topk_weights),
                                   1 if weighted else 0, T, H, K, E, R, _p(dst_row), _p(tokens),
                                   n if tokens is not None else 0, _p(out))
    return out[:n], status


def expanded_rows(topk_idx, E, expert_offset):
    """Expanded row of every (t, k) (see ep_oracle_expanded_rows): int32 [T, K], -1 if masked."""
    lib = _load()
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    expert_offset = np.ascontiguousarray(expert_offset, dtype=np.int32)
    out = np.zeros((T, K), np.int32)
    scratch = np.zeros(max(E, 1), np.int32)
    status = lib.ep_oracle_expanded_rows(_p(topk_idx), T, K, E, _p(expert_offset), _p(out), _p(scratch))
    return out, status


def dispatch_expanded(x_bits, topk_weights, expanded_row, capacity, fp8=False, sf_col_major=False,
                      sf_stride=None, sf_fill=0.0):
    """Expanded dispatch (see ep_oracle_dispatch_expanded); arrays sized by capacity.

    FP8 scales come back as [capacity, H/128] (row-major) or, with
    ``sf_col_major``, as the flat column-major array of H/128 columns of
    ``sf_stride`` entries (default: capacity).  Entries no row writes (expert
    padding rows, the stride's tail) keep ``sf_fill``.
    """
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    expanded_row = np.ascontiguousarray(expanded_row, dtype=np.int32)
    K = expanded_row.shape[1]
    n = max(int(capacity), 1)
    row_bytes = H if fp8 else 2 * H
    nb = H // 128
    if sf_stride is None:
        sf_stride = int(capacity)
    assert sf_stride >= capacity
    recv_x = np.zeros((n, row_bytes), np.uint8)
    recv_sf = None
    if fp8:
        recv_sf = np.full(max(nb * sf_stride, 1) if sf_col_major else n * nb, sf_fill, np.float32)
    recv_src_idx = np.full(n, -1, np.int32)
    recv_weight = np.zeros(n, np.float32)
    status = lib.ep_oracle_dispatch_expanded(_p(x_bits), _p(topk_weights), T, H, K, _p(expanded_row),
                                             int(capacity), 1 if fp8 else 0, 1 if sf_col_major else 0,
                                             int(sf_stride), _p(recv_x), _p(recv_sf),
                                             _p(recv_src_idx), _p(recv_weight))
    res = dict(recv_x=recv_x[:capacity], recv_src_idx=recv_src_idx[:capacity],
               recv_weight=recv_weight[:capacity], status=status)
    if fp8:
        res["recv_sf"] = recv_sf[:nb * sf_stride] if sf_col_major else recv_sf.reshape(n, nb)[:capacity]
    return res


def combine_expanded(y_bits, topk_weights, expanded_row, weighted=True):
    """Expanded combine (see ep_oracle_combine_expanded); float64 [T, H]."""
    lib = _load()
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    expanded_row = np.ascontiguousarray(expanded_row, dtype=np.int32)
    T, K = expanded_row.shape
    H = y_bits.shape[1]
    if topk_weights is None:
        topk_weights = np.zeros((T, K), np.float32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    out = np.zeros((max(T, 1), H), np.float64)
    status = lib.ep_oracle_combine_expanded(_p(y_bits), y_bits.shape[0], _p(topk_weights),
                                            1 if weighted else 0, T, H, K, _p(expanded_row), _p(out))
    return out[:T], status


def combine_topk_weights(recv_topk_weights, dst_row):
    """Combined top-k weights (see ep_oracle_combine_topk_weights): float32 [T, K]."""
    lib = _load()
    rw = np.ascontiguousarray(recv_topk_weights, dtype=np.float32)
    dst_row = np.ascontiguousarray(dst_row, dtype=np.int32)
    T, R = dst_row.shape
    K = rw.shape[1]
    out = np.zeros((max(T, 1), K), np.float32)
    status = lib.ep_oracle_combine_topk_weights(_p(rw), rw.shape[0], T, K, R, _p(dst_row), _p(out))
    return out[:T], status


def accumulate_expert_stats(num_tokens_per_expert, stats):
    """stats (int64, updated in place) += num_tokens_per_expert."""
    lib = _load()
    cnt = np.ascontiguousarray(num_tokens_per_expert, dtype=np.int32)
    assert stats.dtype == np.int64 and stats.flags.c_contiguous
    lib.ep_oracle_accumulate_expert_stats(_p(cnt), cnt.size, _p(stats))
    return stats


def fp8_cast_row(x_bits_row):
    """FP8 e4m3 cast of one bf16 row: returns (codes uint8 [H], sf float32 [H/128])."""
    lib = _load()
    x = np.ascontiguousarray(x_bits_row, dtype=np.uint16)
    H = x.shape[0]
    q = np.zeros(H, np.uint8)
    sf = np.zeros(H // 128, np.float32)
    lib.ep_oracle_fp8_cast_row(_p(x), H, _p(q), _p(sf))
    return q, sf


def e4m3_encode(values):
    """binary32 -> E4M3 codes (RNE, saturating), elementwise, flattened."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).ravel())
    out = np.zeros(v.size, np.uint8)
    lib.ep_oracle_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def e4m3_decode(codes):
    """E4M3 codes -> binary32 values, elementwise, flattened."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8).ravel())
    out = np.zeros(c.size, np.float32)
    lib.ep_oracle_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def float_to_bf16(values):
    """binary32 -> bf16 bit patterns (RNE), elementwise, flattened."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).ravel())
    out = np.zeros(v.size, np.uint16)
    lib.ep_oracle_float_to_bf16_array(_p(v), v.size, _p(out))
    return out


def double_to_bf16(values):
    """float64 -> bf16 bit patterns in one rounding (RNE), elementwise, flattened."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64).ravel())
    out = np.zeros(v.size, np.uint16)
    lib.ep_oracle_double_to_bf16_array(_p(v), v.size, _p(out))
    return out


def node_rows(topk_idx, E, R, ranks_per_node):
    """Rows of the per-node scale-out buffers (see ep_oracle_node_rows):
    returns (node_offset int32 [nodes+1], node_row int32 [T, nodes], status)."""
    lib = _load()
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    nodes = R // ranks_per_node
    node_offset = np.zeros(nodes + 1, np.int32)
    node_row = np.zeros((max(T, 1), nodes), np.int32)
    status = lib.ep_oracle_node_rows(_p(topk_idx), T, K, E, R, ranks_per_node, _p(node_offset), _p(node_row))
    return node_offset, node_row[:T], status


def dispatch_hierarchical(x_bits, topk_idx, topk_weights, E, R, ranks_per_node, node_row, dst_row,
                          node_capacity, recv_capacity, fp8=False, sf_col_major=False, sf_stride=None):
    """Two-stage dispatch (see ep_oracle_dispatch_hierarchical).  Returns the
    node buffers (node_x, node_sf, node_src_idx; unwritten node rows 0 / -1)
    and the receive buffers (recv_*; unwritten rows 0), all sized by the
    capacities."""
    lib = _load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    node_row = np.ascontiguousarray(node_row, dtype=np.int32)
    dst_row = np.ascontiguousarray(dst_row, dtype=np.int32)
    T, H = x_bits.shape
    K = topk_idx.shape[1]
    row_bytes = H if fp8 else 2 * H
    nb = H // 128
    nc, rc = max(int(node_capacity), 1), max(int(recv_capacity), 1)
    if sf_stride is None:
        sf_stride = rc
    node_x = np.zeros((nc, row_bytes), np.uint8)
    node_sf = np.zeros((nc, max(nb, 1)), np.float32)
    node_src_idx = np.full(nc, -1, np.int32)
    recv_x = np.zeros((rc, row_bytes), np.uint8)
    recv_sf = np.zeros(max(nb, 1) * sf_stride if sf_col_major else rc * max(nb, 1), np.float32)
    recv_topk_idx = np.zeros((rc, K), np.int32)
    recv_topk_weights = np.zeros((rc, K), np.float32)
    recv_src_idx = np.zeros(rc, np.int32)
    status = lib.ep_oracle_dispatch_hierarchical(
        _p(x_bits), _p(topk_idx), _p(topk_weights), T, H, K, E, R, ranks_per_node, _p(node_row), _p(dst_row),
        1 if fp8 else 0, int(node_capacity), _p(node_x), _p(node_sf), _p(node_src_idx), int(recv_capacity),
        1 if sf_col_major else 0, sf_stride, _p(recv_x), _p(recv_sf), _p(recv_topk_idx),
        _p(recv_topk_weights), _p(recv_src_idx))
    n, r = int(node_capacity), int(recv_capacity)
    res = dict(node_x=node_x[:n], node_src_idx=node_src_idx[:n], recv_x=recv_x[:r],
               recv_topk_idx=recv_topk_idx[:r], recv_topk_weights=recv_topk_weights[:r],
               recv_src_idx=recv_src_idx[:r], status=status)
    if fp8:
        res["node_sf"] = node_sf[:n]
        res["recv_sf"] = recv_sf if sf_col_major else recv_sf.reshape(rc, nb)[:r]
    return res


def combine_hierarchical(y_bits, topk_idx, topk_weights, E, R, ranks_per_node, node_row, dst_row,
                         node_capacity, weighted=False):
    """Two-stage combine (see ep_oracle_combine_hierarchical): returns
    (node_y uint16 bf16 bits [node_capacity, H], out float64 [T, H], status)."""
    lib = _load()
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = topk_idx.shape
    H = y_bits.shape[1]
    if topk_weights is None:
        topk_weights = np.zeros((T, K), np.float32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    node_row = np.ascontiguousarray(node_row, dtype=np.int32)
    dst_row = np.ascontiguousarray(dst_row, dtype=np.int32)
    nc = max(int(node_capacity), 1)
    node_y = np.zeros((nc, H), np.uint16)
    out = np.zeros((max(T, 1), H), np.float64)
    scratch = np.zeros(max(H, 1), np.float64)
    status = lib.ep_oracle_combine_hierarchical(
        _p(y_bits), y_bits.shape[0], _p(topk_idx), _p(topk_weights), 1 if weighted else 0, T, H, K, E, R,
        ranks_per_node, _p(node_row), _p(dst_row), int(node_capacity), _p(node_y), _p(out), _p(scratch))
    return node_y[:int(node_capacity)], out[:T], status


def bf16_to_float(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def expected_ranks_per_token(E, K, R):
    """Expected number of distinct ranks a token reaches when it picks K
    distinct experts uniformly among E, E/R experts per rank: the
    ``get_expected_topk(num_groups)`` helper of the ``get_theoretical_num_sms``
    fragment of "DeepEP V2 ElasticBuffer architecture" with num_groups = R,
    R * (1 - C(E - E/R, K) / C(E, K)) (exact binomials, one float division)."""
    return R * (1 - math.comb(E - E // R, K) / math.comb(E, K))


def theoretical_num_sms(H, K, E, R, hbm_gbs, fp8=False, combine=False, sm_read_gbs=200.0,
                        sm_write_gbs=50.0, prefer_overlap=True, device_sms=152):
    """The SM count rule of the ``get_theoretical_num_sms`` fragment ("DeepEP
    V2 ElasticBuffer architecture"), read for ranks that share one HBM: the
    bounding link is the HBM, whose traffic is everything the SMs read and
    write.  Steps in the fragment's order:

    1. bandwidth of the bounding link: hbm_gbs;
    2. expected ranks per token g (``expected_ranks_per_token``);
    3. traffic per token: dispatch reads the 2H-byte source row and writes g
       rows (2H bytes bf16, H + 4H/128 FP8); combine reads g bf16 rows and
       writes one;
    4. the link is the bottleneck: time per token = (read + write) / hbm_gbs;
    5. SMs to read / write at sm_read_gbs / sm_write_gbs per SM in that time,
       the larger of the two, x 1.25, at least 4, rounded up to even, at least
       64 unless overlapping with compute, at most device_sms.

    Returns (count, n) with n the unrounded count of step 5."""
    g = expected_ranks_per_token(E, K, R)
    row = (H + 4 * (H // 128)) if fp8 and not combine else 2 * H
    if combine:
        read, write = g * 2 * H, 2 * H
    else:
        read, write = 2 * H, g * row
    traffic = read + write
    n = max(hbm_gbs / traffic * read / sm_read_gbs, hbm_gbs / traffic * write / sm_write_gbs)
    count = max(4, math.ceil(n * 1.25))
    count = (count + 1) // 2 * 2
    if not prefer_overlap:
        count = max(count, 64)
    return min(count, device_sms), n
