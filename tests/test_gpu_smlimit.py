"""SM-limited mode (num_sms > 0: a persistent grid of num_sms CTAs that loop
over the work) must give exactly the default mode's results, for bf16 and FP8
dispatch, unweighted and weighted combine and the expanded variants; one case
is also checked against the oracle directly."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows

pytestmark = pytest.mark.gpu


def _setup(T, H, E, K, R, seed, mask=0.05, expanded=False):
    from gpu_path import B, to_dev, x_tensor
    d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=mask)
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    lay = B.alloc_layout(T, E, R, K=K if expanded else None)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, 0), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st)
    return d, idx, w, x, lay


def _dispatch(B, x, idx, w, E, R, lay, n, H, K, fp8, num_sms, expanded):
    rx = torch.zeros((n, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
    rsf = torch.zeros((n * (H // 128),), dtype=torch.float32, device="cuda") if fp8 else None
    rs = torch.zeros((n,), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dt = B.EP_FP8_E4M3 if fp8 else B.EP_BF16
    if expanded:
        rw = torch.zeros((n,), dtype=torch.float32, device="cuda")
        B.ep_dispatch_expanded(x, idx, w, E, R, lay, rx, rs, rw, st, recv_sf=rsf, out_dtype=dt, num_sms=num_sms)
        extra = [rw]
    else:
        ri = torch.zeros((n, K), dtype=torch.int32, device="cuda")
        rw = torch.zeros((n, K), dtype=torch.float32, device="cuda")
        B.ep_dispatch(x, idx, w, E, R, lay, rx, ri, rw, rs, st, recv_sf=rsf, out_dtype=dt, num_sms=num_sms)
        extra = [ri, rw]
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    out = [rx.view(torch.uint8) if fp8 else rx.view(torch.int16), rs] + extra
    if fp8:
        out.append(rsf)
    return out


@pytest.mark.parametrize("expanded", [False, True])
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("num_sms", [1, 7, 64])
def test_dispatch_sm_limited_matches_default(expanded, fp8, num_sms):
    from gpu_path import B
    T, H, E, K, R = 700, 1024, 64, 6, 8
    d, idx, w, x, lay = _setup(T, H, E, K, R, seed=3, expanded=expanded)
    n = int(lay.expert_offset[-1].item()) if expanded else lay.num_recv
    ref = _dispatch(B, x, idx, w, E, R, lay, n, H, K, fp8, 0, expanded)
    got = _dispatch(B, x, idx, w, E, R, lay, n, H, K, fp8, num_sms, expanded)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("expanded", [False, True])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("num_sms", [1, 7, 64])
def test_combine_sm_limited_matches_default(expanded, weighted, num_sms):
    from gpu_path import B, x_tensor
    T, H, E, K, R = 700, 1024, 64, 6, 8
    d, idx, w, x, lay = _setup(T, H, E, K, R, seed=4, expanded=expanded)
    n = int(lay.expert_offset[-1].item()) if expanded else lay.num_recv
    y = x_tensor(make_rows(n, H, seed=5))
    outs = []
    for ns in (0, num_sms):
        out = torch.full((T, H), 3.0, dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if expanded:
            B.ep_combine_expanded(y, w if weighted else None, K, E, R, lay, out, st, num_sms=ns)
        else:
            B.ep_combine(y, idx, w if weighted else None, E, R, lay, out, st, num_sms=ns)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append(out.view(torch.int16))
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("T,H,E,K,R,num_sms", [
    (300, 7168, 256, 32, 64, 5),    # 32 rows per item: 1 KB pieces
    (257, 4104, 64, 4, 16, 3),      # 8 KB pieces, a 16-byte last piece
    (40, 16, 8, 2, 4, 2),           # rows shorter than a piece
])
def test_combine_ring_shapes_and_empty_tokens(T, H, E, K, R, num_sms):
    """The SM-limited combine (shared-memory ring) against the oracle, with
    tokens whose entries are all masked (items without source rows)."""
    from gpu_path import B, bf16_bits, to_dev, x_tensor
    from tolerance import check_close, rank_combine_bounds
    d = make_inputs(T, H, E, K, R, seed=T + K, mask_frac=0.1, with_x=False)
    d["topk_idx"][[0, T // 2, T - 1]] = -1
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    lay = B.alloc_layout(T, E, R)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, 0), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st)
    n = lay.num_recv
    y_bits = make_rows(n, H, seed=T + 1)
    L = oracle.layout(d["topk_idx"], E, R)
    for weighted in (False, True):
        out = torch.full((T, H), 3.0, dtype=torch.bfloat16, device="cuda")
        st.zero_()
        B.ep_combine(x_tensor(y_bits), idx, w if weighted else None, E, R, lay, out, st, num_sms=num_sms)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref, _ = oracle.combine(y_bits, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted=weighted)
        loose, tight = rank_combine_bounds(y_bits, d["topk_idx"], d["topk_weights"], E, R, L.dst_row, weighted,
                                           ref)
        check_close(bf16_bits(out), ref, loose, tight)
        assert (bf16_bits(out)[[0, T // 2, T - 1]] == 0).all()


def test_sm_limited_against_oracle():
    from gpu_path import B, bf16_bits
    T, H, E, K, R = 1000, 7168, 256, 8, 8
    d, idx, w, x, lay = _setup(T, H, E, K, R, seed=6, mask=0.0)
    n = lay.num_recv
    got = _dispatch(B, x, idx, w, E, R, lay, n, H, K, False, 16, False)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    np.testing.assert_array_equal(got[0].cpu().numpy().view(np.uint16), o["recv_x"].view(np.uint16))
    np.testing.assert_array_equal(got[1].cpu().numpy(), o["recv_src_idx"])
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine(got[0].view(torch.bfloat16), idx, None, E, R, lay, out, st, num_sms=16)
    torch.cuda.synchronize()
    nt = L.is_token_in_rank.sum(axis=1)
    want = (x.float() * torch.from_numpy(nt).cuda().float()[:, None]).to(torch.bfloat16)
    assert torch.equal(out.float(), want.float())


@pytest.mark.parametrize("expanded", [False, True])
@pytest.mark.parametrize("num_sms", [16, 100])
def test_fp8_wide_sm_limited_matches_default(expanded, num_sms):
    """FP8 dispatch in the many-token mode (T >= 8 tokens per SM): the
    SM-limited grid gives exactly the default mode's codes, scales and
    metadata."""
    from gpu_path import B
    T, H, E, K, R = 2048, 1024, 64, 6, 8
    d, idx, w, x, lay = _setup(T, H, E, K, R, seed=8, expanded=expanded)
    n = int(lay.expert_offset[-1].item()) if expanded else lay.num_recv
    ref = _dispatch(B, x, idx, w, E, R, lay, n, H, K, True, 0, expanded)
    got = _dispatch(B, x, idx, w, E, R, lay, n, H, K, True, num_sms, expanded)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("num_sms", [3, 40])
@pytest.mark.parametrize("fp8", [False, True])
def test_sm_limited_capacity_overflow(num_sms, fp8):
    """SM-limited dispatch into too few receive rows, and combine from too few
    expert-output rows: the capacity bit is set and every row that fits is
    what the default mode writes."""
    from gpu_path import B, x_tensor
    T, H, E, K, R = 600, 1024, 64, 6, 8
    d, idx, w, x, lay = _setup(T, H, E, K, R, seed=31)
    n = lay.num_recv
    cap = n - 57
    outs = []
    for ns in (0, num_sms):
        rx = torch.zeros((cap, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
        rsf = torch.zeros((cap * (H // 128),), dtype=torch.float32, device="cuda") if fp8 else None
        rs = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.ep_dispatch(x, idx, w, E, R, lay, rx, None, None, rs, st, recv_sf=rsf,
                      out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16, num_sms=ns)
        torch.cuda.synchronize()
        assert int(st.item()) & B.EP_ERR_CAPACITY
        outs.append((rx.view(torch.uint8).clone(), rs.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    y = x_tensor(make_rows(cap, H, seed=32))
    res = []
    for ns in (0, num_sms):
        out = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.ep_combine(y, idx, w, E, R, lay, out, st, num_sms=ns)
        torch.cuda.synchronize()
        assert int(st.item()) & B.EP_ERR_CAPACITY
        res.append(out.view(torch.int16).clone())
    assert torch.equal(res[0], res[1])

