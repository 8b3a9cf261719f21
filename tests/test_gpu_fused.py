"""GPU parity of ep_layout_and_dispatch (layout and dispatch in one call)
against the CPU oracle: every layout array and every dispatched element
bit-exact, on few-token shapes (where the dispatch derives its destination
rows itself and runs beside the layout kernel) and on shapes beyond that
limit (the two kernels one after the other); equal to the separate calls;
capacity overflow and invalid ids flagged as by the separate calls; and a
combine launched right after the call sees the layout (identity closed form).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_config, make_inputs

pytestmark = pytest.mark.gpu


def _fused(d, E, R, fp8=False, sf_col_major=False, capacity=None, rpn=0, align=1):
    from gpu_path import B, to_dev, x_tensor
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    T, K = idx.shape
    H = x.shape[1]
    lay = B.alloc_layout(T, E, R, rpn)
    for t in (lay.num_tokens_per_rank, lay.num_tokens_per_expert, lay.rank_offset, lay.expert_offset,
              lay.dst_row, lay.token_offset):
        t.fill_(-7)
    ws = torch.full((B.ep_layout_workspace_bytes(T, K, E, R, rpn),), 0xA5, dtype=torch.uint8, device="cuda")
    cap = B.ep_recv_capacity_bound(T, K, R) if capacity is None else capacity
    if fp8:
        rx = torch.full((cap, H), 0x55, dtype=torch.uint8, device="cuda")
        stride = (cap + 3) // 4 * 4
        rsf = torch.full((max((H // 128) * (stride if sf_col_major else cap), 1),), -1.0, dtype=torch.float32,
                         device="cuda")
    else:
        rx = torch.full((cap, H), -3.0, dtype=torch.bfloat16, device="cuda")
        rsf = None
    ri = torch.full((cap, K), -9, dtype=torch.int32, device="cuda")
    rw = torch.full((cap, K), -9.0, dtype=torch.float32, device="cuda")
    rs = torch.full((cap,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_layout_and_dispatch(x, idx, w, E, R, lay, ws, rx, ri, rw, rs, st, recv_sf=rsf,
                             out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16, sf_col_major=sf_col_major,
                             ranks_per_node=rpn, expert_alignment=align)
    torch.cuda.synchronize()
    return dict(lay=lay, recv_x=rx, recv_sf=rsf, recv_topk_idx=ri, recv_topk_weights=rw, recv_src_idx=rs,
                status=int(st.item()), cap=cap, x=x, idx=idx, w=w)


def _check(d, E, R, g, fp8=False, sf_col_major=False, rpn=0, align=1):
    from gpu_path import bf16_bits, layout_host
    L = oracle.layout(d["topk_idx"], E, R, rpn, align)
    got = layout_host(g["lay"])
    for f in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_offset", "expert_offset",
              "dst_row", "token_offset"):
        np.testing.assert_array_equal(got[f], getattr(L, f), err_msg=f)
    if L.src_dst_count is not None:
        np.testing.assert_array_equal(got["src_dst_count"], L.src_dst_count)
    if rpn:
        np.testing.assert_array_equal(got["num_tokens_per_node"], L.num_tokens_per_node)
    n, cap = L.num_recv, g["cap"]
    H = d["x_bits"].shape[1]
    stride = (cap + 3) // 4 * 4
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row, capacity=cap, fp8=fp8,
                        sf_col_major=sf_col_major, sf_stride=stride)
    assert g["status"] == (L.status | o["status"])
    m = min(n, cap)
    if fp8:
        np.testing.assert_array_equal(g["recv_x"][:m].cpu().numpy(), o["recv_x"][:m])
        nb = H // 128
        sf = g["recv_sf"].cpu().numpy()
        if sf_col_major:
            np.testing.assert_array_equal(sf[:nb * stride].reshape(nb, stride)[:, :m],
                                          o["recv_sf"][:nb * stride].reshape(nb, stride)[:, :m])
        else:
            np.testing.assert_array_equal(sf[:m * nb].reshape(m, nb), o["recv_sf"][:m])
    else:
        np.testing.assert_array_equal(bf16_bits(g["recv_x"][:m]).view(np.uint8).reshape(m, 2 * H), o["recv_x"][:m])
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(g[k][:m].cpu().numpy(), o[k][:m], err_msg=k)
    # rows the layout does not use are untouched
    if cap > n:
        assert (g["recv_src_idx"][n:] == -9).all()


@pytest.mark.parametrize("name", ["tiny", "decode"])
@pytest.mark.parametrize("sf_col_major", [False, True])
def test_fused_workloads(name, sf_col_major):
    d = make_config(name)
    c = d["cfg"]
    if sf_col_major and not c.fp8:
        pytest.skip("column-major scales are an FP8 layout")
    g = _fused(d, c.E, c.R, fp8=c.fp8, sf_col_major=sf_col_major)
    _check(d, c.E, c.R, g, fp8=c.fp8, sf_col_major=sf_col_major)


@pytest.mark.parametrize("T,H,E,K,R,mask,fp8,rpn,align", [
    (1, 7168, 256, 8, 8, 0.0, True, 0, 1),
    (31, 256, 64, 6, 32, 0.1, False, 0, 3),
    (32, 1024, 64, 16, 32, 0.0, True, 4, 1),     # K = 16 and 32 ranks: the self-routing limits
    (33, 512, 16, 4, 1, 0.2, False, 0, 1),       # one rank
    (33, 256, 15, 5, 3, 0.1, True, 0, 1),        # odd number of top-k entries (T*K = 165)
    (7, 128, 16, 3, 4, 0.0, False, 0, 2),        # odd again (21), a few tokens
    (255, 2048, 128, 8, 16, 0.5, True, 8, 7),
    (256, 7168, 256, 8, 8, 0.05, False, 0, 1),   # the largest self-routed token count
    (257, 1024, 256, 8, 8, 0.0, True, 0, 1),     # beyond it: one kernel after the other
    (200, 512, 128, 8, 64, 0.0, False, 0, 1),    # 64 ranks: no self routing
    (100, 256, 256, 20, 32, 0.1, True, 0, 1),    # top-20: no self routing
    (2048, 1024, 64, 6, 8, 0.05, True, 0, 1),    # many tokens (FP8 many-token mode)
    (160, 1024, 64, 2, 8, 0.1, True, 0, 1),      # K = 2 (one lane per token's pair), three pieces
    (96, 2048, 32, 4, 16, 0.0, False, 2, 1),     # K = 4, bf16, four pieces (one metadata array each)
])
def test_fused_shapes(T, H, E, K, R, mask, fp8, rpn, align):
    d = make_inputs(T, H, E, K, R, seed=T * 7 + K, mask_frac=mask)
    g = _fused(d, E, R, fp8=fp8, rpn=rpn, align=align)
    _check(d, E, R, g, fp8=fp8, rpn=rpn, align=align)


def test_fused_duplicates_and_invalid_ids():
    """Duplicate experts inside tokens count once per rank; ids outside
    [-1, E) count for no rank and set the invalid-index bit, as the layout
    defines them."""
    T, H, E, K, R = 150, 512, 64, 8, 16
    d = make_inputs(T, H, E, K, R, seed=77)
    rng = np.random.Generator(np.random.PCG64(78))
    d["topk_idx"] = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    for fp8 in (False, True):
        g = _fused(d, E, R, fp8=fp8)
        assert g["status"] & oracle.EP_ERR_INVALID_INDEX
        _check(d, E, R, g, fp8=fp8)


@pytest.mark.parametrize("fp8", [False, True])
def test_fused_capacity_overflow(fp8):
    T, H, E, K, R = 128, 1024, 64, 6, 16
    d = make_inputs(T, H, E, K, R, seed=91)
    n = oracle.layout(d["topk_idx"], E, R).num_recv
    g = _fused(d, E, R, fp8=fp8, capacity=n - 40)
    assert g["status"] & oracle.EP_ERR_CAPACITY
    _check(d, E, R, g, fp8=fp8)


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_fused_equals_separate_calls(name):
    from gpu_path import run_dispatch, run_layout
    d = make_config(name)
    c = d["cfg"]
    g = _fused(d, c.E, c.R, fp8=c.fp8)
    lay, st = run_layout(g["idx"], c.E, c.R)
    ref = run_dispatch(g["x"], g["idx"], g["w"], c.E, c.R, lay, g["cap"], fp8=c.fp8)
    torch.cuda.synchronize()
    assert torch.equal(lay.dst_row, g["lay"].dst_row)
    for k in ("recv_x", "recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        assert torch.equal(ref[k].view(torch.uint8), g[k].view(torch.uint8)), k
    if c.fp8:
        assert torch.equal(ref["recv_sf"], g["recv_sf"])


def test_combine_right_after_the_fused_call_sees_the_layout():
    """The dispatch completes only after the layout, so a combine launched
    right after the call on the same stream reads the final dst_row: the
    identity round trip gives bf16(n(t) * x[t]) exactly, for every token."""
    from gpu_path import B, to_dev, x_tensor
    d = make_config("tiny")
    c = d["cfg"]
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    T, K = idx.shape
    for rep in range(3):
        lay = B.alloc_layout(T, c.E, c.R)
        lay.dst_row.fill_(-1)          # a stale layout would drop every row
        ws = torch.empty(B.ep_layout_workspace_bytes(T, K, c.E, c.R), dtype=torch.uint8, device="cuda")
        cap = B.ep_recv_capacity_bound(T, K, c.R)
        rx = torch.empty((cap, c.H), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty((T, c.H), dtype=torch.bfloat16, device="cuda")
        B.ep_layout_and_dispatch(x, idx, w, c.E, c.R, lay, ws, rx, None, None, None, st)
        B.ep_combine(rx, idx, None, c.E, c.R, lay, out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        nt = lay.is_token_in_rank.sum(dim=1, dtype=torch.int32).float()
        assert torch.equal(out.float(), (x.float() * nt[:, None]).to(torch.bfloat16).float())


def _random_fused_case(seed):
    """A seeded shape inside the one-kernel limits (T <= 256, R <= 32, K <= 16,
    E <= 2048): token counts around warp and piece edges, K of both top-k
    loaders (powers of two: 16-byte pairs; others: one thread per token),
    bf16 or FP8 of several widths, masks, invalid ids, node groups, alignment."""
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    T = int(rng.choice([1, 2, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 152, 200, 255, 256]))
    R = int(rng.choice([1, 2, 4, 8, 16, 32]))
    E = R * int(rng.choice([1, 2, 4, 8, 16, 64]))
    E = min(E, 2048 - 2048 % R)
    K = int(rng.choice([k for k in (1, 2, 3, 4, 5, 6, 8, 12, 16) if k <= E]))
    fp8 = bool(rng.integers(0, 2))
    H = int(rng.choice([128, 256, 1024, 2048, 7168])) if fp8 else int(rng.choice([8, 64, 256, 1024, 7168]))
    rpn = int(rng.choice([0] + [v for v in (1, 2, 4, 8) if R % v == 0]))
    align = int(rng.choice([1, 1, 3, 16]))
    mask = float(rng.choice([0.0, 0.05, 0.3]))
    col = fp8 and bool(rng.integers(0, 2))
    invalid = bool(rng.integers(0, 4) == 0)
    return T, H, E, K, R, fp8, rpn, align, mask, col, invalid


@pytest.mark.parametrize("seed", range(24))
def test_fused_random(seed):
    T, H, E, K, R, fp8, rpn, align, mask, col, invalid = _random_fused_case(seed)
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    if invalid:   # a few ids outside [-1, E): flagged, skipped, every other row intact
        rng = np.random.Generator(np.random.PCG64(seed))
        flat = d["topk_idx"].reshape(-1)
        pick = rng.choice(flat.size, size=max(1, flat.size // 50), replace=False)
        flat[pick] = rng.choice([-3, -2, E, E + 7], size=pick.size)
    g = _fused(d, E, R, fp8=fp8, sf_col_major=col, rpn=rpn, align=align)
    _check(d, E, R, g, fp8=fp8, sf_col_major=col, rpn=rpn, align=align)
