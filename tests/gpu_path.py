"""Test helpers that run the CUDA path through the C ABI (via the binding).

Nothing here computes a result of the method: it allocates device buffers,
calls ep_get_layout / ep_dispatch / ep_combine, and copies results back.
"""
import numpy as np
import torch

from combine_ep_get_gb300 import build as _build

_build.build()
from combine_ep_get_gb300 import binding as B  # noqa: E402


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def x_tensor(x_bits):
    return to_dev(x_bits.view(np.int16), torch.bfloat16)


def run_layout(topk_idx, E, R, ranks_per_node=0, expert_alignment=1, with_src_dst=True):
    idx = topk_idx if isinstance(topk_idx, torch.Tensor) else to_dev(topk_idx)
    T, K = idx.shape
    lay = B.alloc_layout(T, E, R, ranks_per_node, with_src_dst=with_src_dst)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, ranks_per_node), dtype=torch.uint8,
                     device="cuda")
    # garbage in the workspace must not matter
    ws.fill_(0xA5)
    for t in (lay.num_tokens_per_rank, lay.num_tokens_per_expert, lay.rank_offset,
              lay.expert_offset, lay.dst_row, lay.token_offset):
        t.fill_(-7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, status, ranks_per_node, expert_alignment)
    return lay, status


def layout_host(lay):
    out = {}
    for f in ("num_tokens_per_rank", "num_tokens_per_node", "num_tokens_per_expert",
              "is_token_in_rank", "rank_offset", "expert_offset", "dst_row", "src_dst_count",
              "token_offset"):
        v = getattr(lay, f)
        out[f] = None if v is None else v.cpu().numpy()
    return out


def run_dispatch(x_dev, idx_dev, w_dev, E, R, lay, capacity, fp8=False, sf_col_major=False,
                 with_meta=True):
    T, H = x_dev.shape
    K = idx_dev.shape[1]
    cap = max(int(capacity), 0)
    if fp8:
        recv_x = torch.full((cap, H), 0x55, dtype=torch.uint8, device="cuda")
        sf_stride = (cap + 3) // 4 * 4
        n_sf = (H // 128) * sf_stride if sf_col_major else cap * (H // 128)
        recv_sf = torch.full((max(n_sf, 1),), -1.0, dtype=torch.float32, device="cuda")
    else:
        recv_x = torch.full((cap, H), -3.0, dtype=torch.bfloat16, device="cuda")
        recv_sf = None
    ri = torch.full((cap, K), -9, dtype=torch.int32, device="cuda") if with_meta else None
    rw = torch.full((cap, K), -9.0, dtype=torch.float32, device="cuda") if with_meta else None
    rs = torch.full((cap,), -9, dtype=torch.int32, device="cuda") if with_meta else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_dispatch(x_dev, idx_dev, w_dev, E, R, lay, recv_x, ri, rw, rs, status,
                  recv_sf=recv_sf if fp8 else None, out_dtype=B.EP_FP8_E4M3 if fp8 else B.EP_BF16,
                  sf_col_major=sf_col_major)
    return dict(recv_x=recv_x, recv_sf=recv_sf, recv_topk_idx=ri, recv_topk_weights=rw,
                recv_src_idx=rs, status=status)


def run_combine(y_dev, idx_dev, w_dev, E, R, lay, T, H):
    out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_combine(y_dev, idx_dev, w_dev, E, R, lay, out, status)
    return out, status


def bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
