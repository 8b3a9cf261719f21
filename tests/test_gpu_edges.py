"""Edge cases of the whole path on the GPU: empty input, one rank, one expert
per rank, top-1, invalid ids end to end, host-side argument errors."""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_get_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_empty_tokens_whole_path():
    from gpu_path import run_combine, run_dispatch, run_layout, to_dev
    idx = torch.zeros((0, 8), dtype=torch.int64, device="cuda")
    w = torch.zeros((0, 8), dtype=torch.float32, device="cuda")
    x = torch.zeros((0, 7168), dtype=torch.bfloat16, device="cuda")
    lay, st = run_layout(idx, 256, 8)
    assert lay.num_recv == 0 and int(st.item()) == 0
    assert lay.num_tokens_per_rank.cpu().tolist() == [0] * 8
    assert lay.expert_offset.cpu().tolist() == [0] * 257
    res = run_dispatch(x, idx, w, 256, 8, lay, 0)
    out, st2 = run_combine(torch.zeros((0, 7168), dtype=torch.bfloat16, device="cuda"), idx, None, 256,
                           8, lay, 0, 7168)
    torch.cuda.synchronize()
    assert int(res["status"].item()) == 0 and int(st2.item()) == 0


@pytest.mark.parametrize("T,H,E,K,R", [(513, 1024, 8, 1, 1), (300, 512, 16, 1, 16), (129, 256, 64, 4, 64)])
def test_degenerate_shapes_round_trip(T, H, E, K, R):
    from gpu_path import bf16_bits, run_combine, run_dispatch, run_layout, to_dev, x_tensor
    d = make_inputs(T, H, E, K, R, seed=T + R)
    idx, w = to_dev(d["topk_idx"]), to_dev(d["topk_weights"])
    x = x_tensor(d["x_bits"])
    lay, _ = run_layout(idx, E, R)
    n = lay.num_recv
    res = run_dispatch(x, idx, w, E, R, lay, n)
    L = oracle.layout(d["topk_idx"], E, R)
    o = oracle.dispatch(d["x_bits"], d["topk_idx"], d["topk_weights"], E, R, L.dst_row)
    np.testing.assert_array_equal(res["recv_topk_idx"][:n].cpu().numpy(), o["recv_topk_idx"])
    out, st = run_combine(res["recv_x"], idx, None, E, R, lay, T, H)
    nt = L.is_token_in_rank.sum(axis=1)
    want = (x.float() * torch.from_numpy(nt).cuda().float()[:, None]).to(torch.bfloat16)
    assert torch.equal(out.float(), want.float())     # exact values; zeros compare unsigned


def test_invalid_ids_whole_path():
    from gpu_path import bf16_bits, run_combine, run_dispatch, run_layout, to_dev, x_tensor
    T, H, E, K, R = 600, 512, 64, 6, 8
    d = make_inputs(T, H, E, K, R, seed=31)
    bad = d["topk_idx"].copy()
    bad[5, 2] = E + 3
    bad[400, 0] = -2
    idx, w = to_dev(bad), to_dev(d["topk_weights"])
    lay, st = run_layout(idx, E, R)
    res = run_dispatch(x_tensor(d["x_bits"]), idx, w, E, R, lay, lay.num_recv)
    torch.cuda.synchronize()
    assert int(st.item()) == oracle.EP_ERR_INVALID_INDEX
    L = oracle.layout(bad, E, R)
    o = oracle.dispatch(d["x_bits"], bad, d["topk_weights"], E, R, L.dst_row)
    n = L.num_recv
    np.testing.assert_array_equal(res["recv_topk_idx"][:n].cpu().numpy(), o["recv_topk_idx"])
    np.testing.assert_array_equal(res["recv_topk_weights"][:n].cpu().numpy(), o["recv_topk_weights"])
    np.testing.assert_array_equal(bf16_bits(res["recv_x"][:n]), o["recv_x"].view(np.uint16))


def test_host_errors_raise_before_launch():
    from gpu_path import B, run_layout, to_dev
    idx = to_dev(make_inputs(64, 8, 16, 4, 4, seed=1, with_x=False)["topk_idx"])
    lay, _ = run_layout(idx, 16, 4)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.ep_layout_workspace_bytes(64, 4, 16, 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="invalid_arg"):
        B.ep_get_layout(idx, 15, 4, lay, ws, status)               # R does not divide E
    with pytest.raises(RuntimeError, match="unsupported"):
        B.ep_get_layout(idx, 4096, 4, lay, ws, status)             # E beyond the limit
    x = torch.zeros((64, 12), dtype=torch.bfloat16, device="cuda")  # H % 8 != 0
    rx = torch.zeros((300, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="invalid_arg"):
        B.ep_dispatch(x, idx, None, 16, 4, lay, rx, None, None, None, status)
    big = torch.zeros((65, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="invalid_arg"):         # misaligned x (offset 2 bytes)
        B.ep_dispatch(big.view(-1)[1:1 + 64 * 8].view(64, 8), idx, None, 16, 4, lay,
                      torch.zeros((300, 8), dtype=torch.bfloat16, device="cuda"), None, None, None, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
