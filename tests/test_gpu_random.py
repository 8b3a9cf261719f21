"""Seeded random sweep: layout, dispatch (bf16 or FP8) and combine (weighted
or not) against the CPU oracle on shapes drawn across the supported ranges,
so that every launch path (single-CTA, cluster and tiled layouts; few- and
many-token dispatch and combine) meets ragged sizes, masks, alignments and
node groups it was not tuned on.

Layout, indices and payloads bit-exact; combine within 1e-2 of the sum of
magnitudes (fp32 accumulation, bf16 out)."""
import numpy as np
import pytest

import oracle
from combine_ep_get_gb300.inputs import make_inputs, make_rows

pytestmark = pytest.mark.gpu

N_CASES = 48


def _draw_case(i):
    rng = np.random.Generator(np.random.PCG64(1000 + i))
    R = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 128]))
    epr = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    while R * epr > 2048:
        epr //= 2
    E = R * max(epr, 1)
    K = int(rng.integers(1, min(32, E) + 1))
    base = int(rng.choice([0, 1, 31, 32, 33, 127, 128, 255, 500, 1023, 1024, 1025, 1500]))
    T = max(0, base + int(rng.integers(-1, 2)))
    fp8 = bool(rng.random() < 0.4)
    H = int(rng.choice([128, 256, 384, 1024, 2048])) if fp8 else int(rng.choice([8, 16, 128, 264, 1024, 2048]))
    divisors = [d for d in range(1, R + 1) if R % d == 0]
    rpn = int(rng.choice(divisors)) if rng.random() < 0.4 else 0
    align = int(rng.choice([1, 1, 2, 7, 128]))
    mask = float(rng.choice([0.0, 0.0, 0.1, 0.5]))
    weighted = bool(rng.random() < 0.5)
    return dict(T=T, H=H, E=E, K=K, R=R, rpn=rpn, align=align, mask=mask, fp8=fp8, weighted=weighted,
                seed=2000 + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_layout_dispatch_combine(i):
    from gpu_path import bf16_bits, layout_host, run_combine, run_dispatch, run_layout, to_dev, x_tensor
    from tolerance import check_close, rank_combine_bounds
    c = _draw_case(i)
    T, H, E, K, R = c["T"], c["H"], c["E"], c["K"], c["R"]
    d = make_inputs(T, H, E, K, R, seed=c["seed"], mask_frac=c["mask"])
    idx_h, w_h, x_h = d["topk_idx"], d["topk_weights"], d["x_bits"]
    idx, w = to_dev(idx_h), to_dev(w_h)

    # layout
    lay, st = run_layout(idx, E, R, c["rpn"], c["align"])
    g = layout_host(lay)
    L = oracle.layout(idx_h, E, R, c["rpn"], c["align"])
    for f in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_offset",
              "expert_offset", "dst_row", "token_offset"):
        np.testing.assert_array_equal(g[f], getattr(L, f), err_msg="%s %s" % (f, c))
    if c["rpn"]:
        np.testing.assert_array_equal(g["num_tokens_per_node"], L.num_tokens_per_node, err_msg=str(c))
    if L.src_dst_count is not None:
        np.testing.assert_array_equal(g["src_dst_count"], L.src_dst_count, err_msg=str(c))
    assert int(st.item()) == L.status == 0, c
    n = L.num_recv

    # dispatch
    res = run_dispatch(x_tensor(x_h), idx, w, E, R, lay, n, fp8=c["fp8"])
    assert int(res["status"].item()) == 0, c
    o = oracle.dispatch(x_h, idx_h, w_h, E, R, L.dst_row, fp8=c["fp8"])
    if c["fp8"]:
        np.testing.assert_array_equal(res["recv_x"][:n].cpu().numpy(), o["recv_x"], err_msg=str(c))
        sf = res["recv_sf"].cpu().numpy()[:n * (H // 128)].reshape(n, H // 128)
        np.testing.assert_array_equal(sf, o["recv_sf"], err_msg=str(c))
    else:
        got = bf16_bits(res["recv_x"][:n]).view(np.uint8).reshape(n, 2 * H)   # the oracle's rows are bytes
        np.testing.assert_array_equal(got, o["recv_x"], err_msg=str(c))
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        np.testing.assert_array_equal(res[k][:n].cpu().numpy(), o[k], err_msg="%s %s" % (k, c))

    # combine of stand-in expert outputs
    y_bits = make_rows(n, H, seed=c["seed"] + 1)
    out, st = run_combine(x_tensor(y_bits), idx, w if c["weighted"] else None, E, R, lay, T, H)
    assert int(st.item()) == 0, c
    ref, _ = oracle.combine(y_bits, idx_h, w_h, E, R, L.dst_row, weighted=c["weighted"])
    loose, tight = rank_combine_bounds(y_bits, idx_h, w_h, E, R, L.dst_row, c["weighted"], ref)
    check_close(bf16_bits(out), ref, loose, tight)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_expanded_layout(i):
    """The same shapes with expanded rows (and node rows where there are node
    groups) requested: the whole layout against the oracle."""
    import torch
    from gpu_path import B, layout_host, to_dev
    c = _draw_case(i)
    T, E, K, R = c["T"], c["E"], c["K"], c["R"]
    d = make_inputs(T, 8, E, K, R, seed=c["seed"], mask_frac=c["mask"], with_x=False)
    idx_h = d["topk_idx"]
    lay = B.alloc_layout(T, E, R, c["rpn"], K=K, node_rows=c["rpn"] > 0)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, c["rpn"]), dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)
    lay.expanded_row.fill_(-7)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(to_dev(idx_h), E, R, lay, ws, st, c["rpn"], c["align"])
    torch.cuda.synchronize()
    g = layout_host(lay)
    L = oracle.layout(idx_h, E, R, c["rpn"], c["align"])
    for f in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_offset",
              "expert_offset", "dst_row"):
        np.testing.assert_array_equal(g[f], getattr(L, f), err_msg="%s %s" % (f, c))
    want, _ = oracle.expanded_rows(idx_h, E, L.expert_offset)
    np.testing.assert_array_equal(lay.expanded_row.cpu().numpy(), want, err_msg=str(c))
    if c["rpn"]:
        off, rows, _ = oracle.node_rows(idx_h, E, R, c["rpn"])
        np.testing.assert_array_equal(lay.node_row.cpu().numpy(), rows, err_msg=str(c))
        np.testing.assert_array_equal(lay.node_offset.cpu().numpy(), off, err_msg=str(c))
    assert int(st.item()) == 0, c

