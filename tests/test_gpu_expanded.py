"""GPU parity of the expanded (per-expert) receive layout, dispatch and combine
against the CPU oracle: expanded rows bit-exact (duplicates, masked and invalid
entries, alignment padding, all five workloads at full size), expanded
dispatch payload / source / weight bit-exact (bf16 and FP8), expanded combine
within the combine tolerance and exact for the unweighted identity expert."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_inputs, make_rows
from tolerance import check_close, combine_bounds, expanded_sources

pytestmark = pytest.mark.gpu


def _layout(idx_np, E, R, align=1, rpn=0):
    from gpu_path import B, to_dev
    idx = to_dev(idx_np)
    T, K = idx.shape
    lay = B.alloc_layout(T, E, R, rpn, K=K)
    lay.expanded_row.fill_(-7)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, rpn), dtype=torch.uint8, device="cuda")
    ws.fill_(0x5A)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st, rpn, align)
    return idx, lay, st


def _oracle_rows(idx_np, E, R, align=1):
    L = oracle.layout(idx_np, E, R, 0, align)
    rows, st = oracle.expanded_rows(idx_np, E, L.expert_offset)
    return L, rows, st


@pytest.mark.parametrize("T,K,E,R,align,mode", [
    (128, 4, 16, 4, 1, "uniform"),
    (1000, 8, 256, 8, 128, "masked"),
    (777, 6, 96, 12, 7, "replace"),        # duplicate experts inside tokens
    (513, 5, 40, 8, 3, "invalid"),
    (300, 32, 2048, 1024, 1, "uniform"),   # top-32, 2048 experts
    (1, 8, 256, 8, 4, "uniform"),
])
def test_expanded_rows(T, K, E, R, align, mode):
    rng = np.random.Generator(np.random.PCG64(T + K + E))
    if mode in ("uniform", "masked"):
        idx = make_inputs(T, 8, E, K, R, seed=T, mask_frac=0.2 if mode == "masked" else 0.0,
                          with_x=False)["topk_idx"]
    elif mode == "replace":
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)
    else:
        idx = rng.integers(-3, E + 3, size=(T, K)).astype(np.int64)
    _, lay, st = _layout(idx, E, R, align)
    L, rows, ost = _oracle_rows(idx, E, R, align)
    np.testing.assert_array_equal(lay.expanded_row.cpu().numpy(), rows)
    np.testing.assert_array_equal(lay.expert_offset.cpu().numpy(), L.expert_offset)
    np.testing.assert_array_equal(lay.dst_row.cpu().numpy(), L.dst_row)
    assert int(st.item()) == ost


@pytest.mark.parametrize("name", list(CONFIGS))
def test_expanded_rows_workloads(name):
    d = make_config(name, with_x=False)
    c = d["cfg"]
    _, lay, st = _layout(d["topk_idx"], c.E, c.R, 1, c.ranks_per_node)
    _, rows, _ = _oracle_rows(d["topk_idx"], c.E, c.R, 1)
    np.testing.assert_array_equal(lay.expanded_row.cpu().numpy(), rows)
    assert int(st.item()) == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("T,H,E,K,R,align,mask", [
    (500, 1024, 64, 6, 8, 16, 0.1), (64, 7168, 256, 8, 32, 1, 0.0), (1000, 256, 256, 8, 8, 128, 0.02),
])
def test_expanded_dispatch(fp8, T, H, E, K, R, align, mask):
    _check_expanded_dispatch(fp8, T, H, E, K, R, align, mask, seed=T + H)


def _check_expanded_dispatch(fp8, T, H, E, K, R, align, mask, seed, sf_col_major=False, num_sms=0):
    from gpu_path import B, bf16_bits, x_tensor
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    idx, lay, _ = _layout(d["topk_idx"], E, R, align)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    cap = int(lay.expert_offset[-1].item())
    sf_stride = (cap + 3) // 4 * 4      # the library's column stride: capacity rounded up to 4
    if fp8:
        rx = torch.full((cap, H), 0x55, dtype=torch.uint8, device="cuda")
        n_sf = (H // 128) * sf_stride if sf_col_major else cap * (H // 128)
        rsf = torch.full((max(n_sf, 1),), -1.0, dtype=torch.float32, device="cuda")
    else:
        rx = torch.full((cap, H), -3.0, dtype=torch.bfloat16, device="cuda")
        rsf = None
    rs = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    rw = torch.full((cap,), -9.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_expanded(x_tensor(d["x_bits"]), idx, w, E, R, lay, rx, rs, rw, st, recv_sf=rsf,
                           out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16, sf_col_major=sf_col_major,
                           num_sms=num_sms)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    L, rows, _ = _oracle_rows(d["topk_idx"], E, R, align)
    o = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], rows, cap, fp8=fp8, sf_col_major=sf_col_major,
                                 sf_stride=sf_stride, sf_fill=-1.0)
    valid = np.unique(rows[rows >= 0])
    gx = rx.cpu().numpy() if fp8 else bf16_bits(rx).view(np.uint8).reshape(cap, 2 * H)
    np.testing.assert_array_equal(gx[valid], o["recv_x"][valid])
    np.testing.assert_array_equal(rs.cpu().numpy(), o["recv_src_idx"])       # padding stays -1
    np.testing.assert_array_equal(rw.cpu().numpy()[valid], o["recv_weight"][valid])
    if fp8 and sf_col_major:
        # the whole column-major array: written rows' scales, and the fill of
        # padding rows and of the stride's tail, untouched
        np.testing.assert_array_equal(rsf.cpu().numpy()[:(H // 128) * sf_stride], o["recv_sf"])
    elif fp8:
        np.testing.assert_array_equal(rsf.cpu().numpy()[:cap * (H // 128)].reshape(cap, H // 128)[valid],
                                      o["recv_sf"][valid])


@pytest.mark.parametrize("T,H,E,K,R,align,mask,num_sms", [
    (64, 7168, 256, 8, 32, 1, 0.0, 0),        # few-token lane mode (16 lanes per block)
    (500, 1024, 64, 6, 8, 16, 0.1, 0),        # expert padding rows inside the scale columns
    (1000, 256, 256, 8, 8, 128, 0.02, 0),     # mostly padding (alignment 128)
    (2048, 1024, 64, 6, 8, 4, 0.05, 0),       # many-token lane mode (8 lanes per block)
    (2048, 1024, 64, 6, 8, 4, 0.05, 16),      # SM-limited, many-token
    (333, 2048, 96, 5, 12, 7, 0.1, 36),       # SM-limited, few-token, odd alignment
    (3, 128, 16, 4, 4, 3, 0.0, 0),            # capacity not a multiple of 4: ragged stride tail
])
def test_expanded_dispatch_fp8_col_major(T, H, E, K, R, align, mask, num_sms):
    """Expanded FP8 dispatch with TMA-aligned column-major scales (stride =
    capacity rounded up to 4) against the oracle, element by element over the
    whole scale array."""
    _check_expanded_dispatch(True, T, H, E, K, R, align, mask, seed=T + 3 * H, sf_col_major=True, num_sms=num_sms)


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("T,H,E,K,R,align,mask", [
    (500, 1024, 64, 6, 8, 16, 0.1), (4096, 7168, 256, 8, 8, 1, 0.0), (200, 256, 2048, 32, 1024, 4, 0.1),
])
def test_expanded_combine(weighted, T, H, E, K, R, align, mask):
    _check_expanded_combine(weighted, T, H, E, K, R, align, mask, seed=T + 2 * H)


def _check_expanded_combine(weighted, T, H, E, K, R, align, mask, seed):
    from gpu_path import B, bf16_bits, x_tensor
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask, with_x=False)
    idx, lay, _ = _layout(d["topk_idx"], E, R, align)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    cap = int(lay.expert_offset[-1].item())
    y_bits = make_rows(cap, H, seed=T + 1)
    out = torch.full((T, H), 5.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine_expanded(x_tensor(y_bits), w if weighted else None, K, E, R, lay, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, rows, _ = _oracle_rows(d["topk_idx"], E, R, align)
    toks = np.arange(T) if T <= 1000 else np.unique(np.concatenate([[0, T - 1], np.arange(0, T, 97)]))
    ref, _ = oracle.combine_expanded(y_bits, d["topk_weights"][toks], rows[toks], weighted=weighted)
    srows, c, a, m = expanded_sources(rows, d["topk_weights"], weighted, tokens=toks)
    loose, tight = combine_bounds(y_bits, srows, c, a, ref, m)
    check_close(bf16_bits(out)[toks], ref, loose, tight)


def test_expanded_round_trip_closed_form():
    """expanded dispatch -> identity expert -> unweighted expanded combine
    == bf16(valid_slots(t) * x[t]) exactly, on the DeepSeek-V3-shaped workload."""
    from gpu_path import B, x_tensor
    d = make_config("dsv3")
    c = d["cfg"]
    idx, lay, _ = _layout(d["topk_idx"], c.E, c.R, 1)
    x = x_tensor(d["x_bits"])
    w = torch.from_numpy(d["topk_weights"]).cuda()
    cap = int(lay.expert_offset[-1].item())
    rx = torch.empty((cap, c.H), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_expanded(x, idx, w, c.E, c.R, lay, rx, None, None, st)
    out = torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda")
    B.ep_combine_expanded(rx, None, c.K, c.E, c.R, lay, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n_valid = (idx >= 0).sum(dim=1).float()
    want = (x.float() * n_valid[:, None]).to(torch.bfloat16)
    assert torch.equal(out.float(), want.float())


def test_expanded_dispatch_fp8_wide():
    """Expanded FP8 dispatch in the many-token mode against the oracle."""
    from gpu_path import B, x_tensor
    T, H, E, K, R = 2048, 1024, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=19, mask_frac=0.05)
    idx, lay, _ = _layout(d["topk_idx"], E, R, 1)
    w = torch.from_numpy(d["topk_weights"]).cuda()
    cap = int(lay.expert_offset[-1].item())
    rx = torch.full((cap, H), 0x55, dtype=torch.uint8, device="cuda")
    rsf = torch.full((cap * (H // 128),), -1.0, dtype=torch.float32, device="cuda")
    rs = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
    rw = torch.full((cap,), -9.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch_expanded(x_tensor(d["x_bits"]), idx, w, E, R, lay, rx, rs, rw, st, recv_sf=rsf,
                           out_dtype=B.EP_FP8_E4M3)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, rows, _ = _oracle_rows(d["topk_idx"], E, R, 1)
    o = oracle.dispatch_expanded(d["x_bits"], d["topk_weights"], rows, cap, fp8=True)
    valid = np.unique(rows[rows >= 0])
    np.testing.assert_array_equal(rx.cpu().numpy()[valid], o["recv_x"][valid])
    np.testing.assert_array_equal(rsf.cpu().numpy().reshape(cap, H // 128)[valid], o["recv_sf"][valid])
    np.testing.assert_array_equal(rs.cpu().numpy(), o["recv_src_idx"])


@pytest.mark.parametrize("i", range(24))
def test_random_expanded_dispatch_combine(i):
    """Expanded dispatch (FP8 cases alternate row- and column-major scales)
    and weighted / unweighted combine on the random sweep's shapes and
    alignments."""
    from test_gpu_random import _draw_case
    c = _draw_case(i)
    _check_expanded_dispatch(c["fp8"], c["T"], c["H"], c["E"], c["K"], c["R"], c["align"], c["mask"], seed=c["seed"],
                             sf_col_major=c["fp8"] and i % 2 == 1)
    _check_expanded_combine(c["weighted"], c["T"], c["H"], c["E"], c["K"], c["R"], c["align"], c["mask"],
                            seed=c["seed"] + 3)

