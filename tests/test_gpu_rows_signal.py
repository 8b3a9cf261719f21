"""The rows-ready signal of ep_layout_and_dispatch on the cluster layout path.

Each CTA of the one-cluster layout kernel publishes a per-call tag in a line
of the caller's workspace once its block of dst_row is written; the dispatch
CTAs of those tokens start on that tag instead of on the layout kernel's
completion (the CTAs of the first wave, which start while the layout kernel
runs), count themselves, and the grid's last CTA clears the tags.  Checked
here, all bit for bit against the separate calls (ep_get_layout, then
ep_dispatch), which share no signal:
- the DeepSeek-V3-shaped and skewed workloads, bf16 and FP8;
- after a call, no slot line holds a tag;
- several routings through one workspace, one after the other;
- a CUDA graph of the call replayed on new routing (the same tag on every
  replay);
- a test-only library whose poll gives up at once, so that the CTAs take
  the fallback (the layout kernel's completion).
"""
import ctypes

import pytest
import torch

from combine_ep_get_gb300.inputs import make_config, make_inputs

pytestmark = pytest.mark.gpu

READY_WORDS = 16   # 64-bit words per slot line


def _cluster_plan(T):
    """CTAs and tokens per CTA of the one-cluster layout: one CTA per 256
    tokens, at most 16, ranges of whole 32-token words."""
    ctas = min(max((T + 255) // 256, 1), 16)
    tpc = max(((T + ctas - 1) // ctas + 31) // 32 * 32, 32)
    return (T + tpc - 1) // tpc, tpc


def _buffers(T, H, K, E, R, fp8):
    from gpu_path import B
    lay = B.alloc_layout(T, E, R, 0)
    for t in (lay.num_tokens_per_rank, lay.num_tokens_per_expert, lay.rank_offset, lay.expert_offset,
              lay.dst_row, lay.token_offset):
        t.fill_(-7)
    ws = torch.full((B.ep_layout_workspace_bytes(T, K, E, R, 0),), 0xA5, dtype=torch.uint8, device="cuda")
    cap = B.ep_recv_capacity_bound(T, K, R)
    if fp8:
        rx = torch.full((cap, H), 0x55, dtype=torch.uint8, device="cuda")
        rsf = torch.full((cap * (H // 128),), -1.0, dtype=torch.float32, device="cuda")
    else:
        rx = torch.full((cap, H), -3.0, dtype=torch.bfloat16, device="cuda")
        rsf = None
    return dict(lay=lay, ws=ws, cap=cap, recv_x=rx, recv_sf=rsf,
                recv_topk_idx=torch.full((cap, K), -9, dtype=torch.int32, device="cuda"),
                recv_topk_weights=torch.full((cap, K), -9.0, dtype=torch.float32, device="cuda"),
                recv_src_idx=torch.full((cap,), -9, dtype=torch.int32, device="cuda"),
                status=torch.zeros(1, dtype=torch.int32, device="cuda"))


def _fused_call(b, x, idx, w, E, R, fp8, lib=None):
    from gpu_path import B
    if lib is None:
        B.ep_layout_and_dispatch(x, idx, w, E, R, b["lay"], b["ws"], b["recv_x"], b["recv_topk_idx"],
                                 b["recv_topk_weights"], b["recv_src_idx"], b["status"], recv_sf=b["recv_sf"],
                                 out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16)
        return
    T, H = x.shape
    K = idx.shape[1]
    p = lambda t: None if t is None else t.data_ptr()   # noqa: E731
    code = lib.ep_layout_and_dispatch(p(x), p(idx), p(w), T, H, K, E, R, 0, 1, ctypes.byref(b["lay"].c),
                                      p(b["ws"]), b["ws"].numel(), B.EP_FP8_E4M3 if fp8 else B.EP_BF16, b["cap"],
                                      p(b["recv_x"]), p(b["recv_sf"]), 0, p(b["recv_topk_idx"]),
                                      p(b["recv_topk_weights"]), p(b["recv_src_idx"]), p(b["status"]),
                                      torch.cuda.current_stream().cuda_stream)
    assert code == B.EP_OK


def _separate(x, idx, w, E, R, cap, fp8):
    from gpu_path import run_dispatch, run_layout
    lay, st = run_layout(idx, E, R)
    res = run_dispatch(x, idx, w, E, R, lay, cap, fp8=fp8)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return lay, res


def _assert_same(b, lay, res, H, fp8):
    for f in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "rank_offset", "expert_offset",
              "dst_row", "token_offset", "src_dst_count"):
        assert torch.equal(getattr(b["lay"], f), getattr(lay, f)), f
    n = int(lay.rank_offset[-1].item())
    assert n > 0
    assert int(b["status"].item()) == int(res["status"].item())
    if fp8:
        assert torch.equal(b["recv_x"][:n], res["recv_x"][:n])
        assert torch.equal(b["recv_sf"][:n * (H // 128)], res["recv_sf"][:n * (H // 128)])
    else:
        assert torch.equal(b["recv_x"][:n].view(torch.int16), res["recv_x"][:n].view(torch.int16))
    for k in ("recv_topk_idx", "recv_topk_weights", "recv_src_idx"):
        assert torch.equal(b[k][:n], res[k][:n]), k


def _assert_slots_clear(ws, T):
    """No line holds a tag after the call.  The readers are the dispatch
    CTAs of the first wave (the lowest item numbers, token by token), so the
    lines count all the pieces of their tokens, then one line part of them,
    then none."""
    C, tpc = _cluster_plan(T)
    w64 = ws.view(torch.int64).cpu().numpy()
    w32 = ws.view(torch.int32).cpu().numpy()
    for c in range(C):
        assert w64[c * READY_WORDS] == 0, c
    counts = [int(w32[c * 2 * READY_WORDS + 2]) for c in range(C)]
    assert counts[0] > 0, counts
    assert all(a >= b for a, b in zip(counts, counts[1:])), counts
    assert len([n for n in counts if 0 < n < counts[0]]) <= 1, counts


@pytest.mark.parametrize("name,fp8", [("dsv3", False), ("dsv3", True), ("skewed", False)])
def test_cluster_path_equals_separate_calls(name, fp8):
    from gpu_path import to_dev, x_tensor
    d = make_config(name)
    c = d["cfg"]
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    T, H = x.shape
    b = _buffers(T, H, idx.shape[1], c.E, c.R, fp8)
    _fused_call(b, x, idx, w, c.E, c.R, fp8)
    torch.cuda.synchronize()
    lay, res = _separate(x, idx, w, c.E, c.R, b["cap"], fp8)
    _assert_same(b, lay, res, H, fp8)
    _assert_slots_clear(b["ws"], T)


@pytest.mark.parametrize("fp8", [False, True])
def test_several_routings_through_one_workspace(fp8):
    from gpu_path import to_dev, x_tensor
    T, H, E, K, R = 2048, 1024, 64, 6, 8          # 8 layout CTAs; FP8 in the many-token mode
    b = None
    for seed in (21, 22, 23):
        d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=0.05 * (seed - 21))
        idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
        if b is None:
            b = _buffers(T, H, K, E, R, fp8)
        _fused_call(b, x, idx, w, E, R, fp8)
        torch.cuda.synchronize()
        lay, res = _separate(x, idx, w, E, R, b["cap"], fp8)
        _assert_same(b, lay, res, H, fp8)
        _assert_slots_clear(b["ws"], T)


@pytest.mark.parametrize("fp8", [False, True])
def test_graph_replays_on_new_routing(fp8):
    from gpu_path import to_dev, x_tensor
    T, H, E, K, R = 4096, 2048, 256, 8, 8         # 16 layout CTAs
    d0 = make_inputs(T, H, E, K, R, seed=30)
    idx, w, x = to_dev(d0["topk_idx"]), to_dev(d0["topk_weights"]), x_tensor(d0["x_bits"])
    b = _buffers(T, H, K, E, R, fp8)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fused_call(b, x, idx, w, E, R, fp8)      # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _fused_call(b, x, idx, w, E, R, fp8)
    for seed in (31, 32, 33):
        d = make_inputs(T, H, E, K, R, seed=seed, mask_frac=0.1)
        idx.copy_(to_dev(d["topk_idx"]))
        w.copy_(to_dev(d["topk_weights"]))
        x.copy_(x_tensor(d["x_bits"]))
        b["status"].zero_()
        g.replay()
        torch.cuda.synchronize()
        lay, res = _separate(x, idx, w, E, R, b["cap"], fp8)
        _assert_same(b, lay, res, H, fp8)
        _assert_slots_clear(b["ws"], T)


@pytest.mark.parametrize("fp8", [False, True])
def test_fallback_when_the_poll_gives_up(fp8):
    """A test-only library whose poll stops after its first look: the CTAs
    that find no tag wait for the layout kernel's completion, then count
    themselves as readers like the others, and the last CTA clears the
    tags as usual."""
    from combine_ep_get_gb300 import build
    from gpu_path import B, to_dev, x_tensor
    path = build.build_variant("rowswait0", ["-DEP_ROWS_WAIT_NS=0ull"])
    lib = ctypes.CDLL(path)
    lib.ep_layout_and_dispatch.restype = B.library().ep_layout_and_dispatch.restype
    lib.ep_layout_and_dispatch.argtypes = B.library().ep_layout_and_dispatch.argtypes
    d = make_config("dsv3")
    c = d["cfg"]
    idx, w, x = to_dev(d["topk_idx"]), to_dev(d["topk_weights"]), x_tensor(d["x_bits"])
    T, H = x.shape
    b = _buffers(T, H, idx.shape[1], c.E, c.R, fp8)
    for _ in range(2):
        _fused_call(b, x, idx, w, c.E, c.R, fp8, lib=lib)
        torch.cuda.synchronize()
        _assert_slots_clear(b["ws"], T)
    lay, res = _separate(x, idx, w, c.E, c.R, b["cap"], fp8)
    _assert_same(b, lay, res, H, fp8)
