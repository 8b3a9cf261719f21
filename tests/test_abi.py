"""The C ABI library on a machine without a GPU: it loads, exports every
function include/ep_get.h declares, and its host-side checks reject bad
arguments with the documented codes before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep_get.h")


@pytest.fixture(scope="module")
def lib():
    from combine_ep_get_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n.startswith("ep_")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ep_get_layout", "ep_dispatch", "ep_combine", "ep_layout_workspace_bytes",
              "ep_recv_capacity_bound", "ep_status_string", "ep_abi_version", "ep_dispatch_expanded",
              "ep_combine_expanded", "ep_expanded_capacity_bound", "ep_combine_topk_weights",
              "ep_accumulate_expert_stats", "ep_theoretical_num_sms",
              "ep_dispatch_hierarchical", "ep_combine_hierarchical", "ep_layout_and_dispatch",
              "ep_bounds_checked"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings_and_sizes(lib):
    lib.ep_status_string.restype = ctypes.c_char_p
    assert lib.ep_status_string(0) == b"ok"
    assert lib.ep_status_string(4 | 8) == b"invalid_index|capacity"
    assert lib.ep_status_string(999) == b"unknown"
    assert lib.ep_status_string(64 | 16) == b"timeout|out_of_bounds"
    lib.ep_recv_capacity_bound.restype = ctypes.c_int64
    assert lib.ep_recv_capacity_bound(4096, 8, 8) == 4096 * 8
    assert lib.ep_recv_capacity_bound(128, 8, 4) == 512
    lib.ep_layout_workspace_bytes.restype = ctypes.c_size_t
    ws = lib.ep_layout_workspace_bytes(4096, 8, 256, 8, 0)
    tiles = 16
    assert ws >= 4 * tiles * (8 + 256 + 8 * 8)
    assert lib.ep_abi_version() == 8
    assert lib.ep_bounds_checked() == 0   # the product library


def test_host_checks_reject_before_any_launch(lib):
    """Every call below fails a host check, so no CUDA call is made."""
    from combine_ep_get_gb300 import binding as B
    L = B.ep_layout_t()
    vp = ctypes.c_void_p
    st = vp(16)            # a stand-in device address; never dereferenced on these paths
    # layout: null out / status, bad shapes, limits
    f = lib.ep_get_layout
    f.restype = ctypes.c_int32
    f.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.POINTER(B.ep_layout_t), vp, ctypes.c_size_t, vp, vp]
    assert f(None, 10, 8, 256, 8, 0, 1, None, None, 0, st, None) == B.EP_ERR_INVALID_ARG
    assert f(None, 10, 8, 256, 7, 0, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_INVALID_ARG
    assert f(None, 10, 8, 4096, 8, 0, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_UNSUPPORTED
    assert f(None, 10, 33, 256, 8, 0, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_UNSUPPORTED
    assert f(None, 10, 8, 2048, 4, 0, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_UNSUPPORTED
    assert f(None, -1, 8, 256, 8, 0, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_INVALID_ARG
    assert f(None, 10, 8, 256, 8, 3, 1, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_INVALID_ARG
    assert f(None, 10, 8, 256, 8, 0, 0, ctypes.byref(L), None, 0, st, None) == B.EP_ERR_INVALID_ARG
    # layout: arrays missing / misaligned
    L2 = B.ep_layout_t(16, None, 32, 48, 64, 80, 96, None, None)
    assert f(vp(16), 10, 8, 256, 8, 0, 1, ctypes.byref(L2), None, 0, st, None) == B.EP_ERR_INVALID_ARG
    L3 = B.ep_layout_t(16, None, 32, 48, 64, 80, 97, None, None)      # dst_row misaligned
    assert f(vp(16), 10, 8, 256, 8, 0, 1, ctypes.byref(L3), vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG
    # workspace too small
    assert f(vp(16), 10, 8, 256, 8, 0, 1, ctypes.byref(L2), vp(256), 8, st, None) == B.EP_ERR_INVALID_ARG
    # src_dst_count needs R | T
    L4 = B.ep_layout_t(16, None, 32, 48, 64, 80, 96, 112, None)
    assert f(vp(16), 10, 8, 256, 8, 0, 1, ctypes.byref(L4), vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG
    # dispatch
    d = lib.ep_dispatch
    d.restype = ctypes.c_int32
    d.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.POINTER(B.ep_layout_t), ctypes.c_int, ctypes.c_int64, vp, vp, ctypes.c_int,
                  vp, vp, vp, ctypes.c_int, vp, vp]
    args = [vp(16), vp(32), vp(48), 10, 7168, 8, 256, 8, ctypes.byref(L2), B.EP_BF16, 100,
            vp(64), None, 0, None, None, None, 0, st, None]
    bad = list(args); bad[4] = 7164                      # H % 8
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[9] = B.EP_FP8_E4M3; bad[4] = 7168 + 64   # H % 128 for FP8
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[9] = B.EP_FP8_E4M3             # FP8 needs recv_sf
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[9] = 7                         # unknown dtype
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[0] = vp(18)                    # x misaligned
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[10] = -1                       # capacity
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[11] = None                     # recv_x missing
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[15] = vp(80); bad[2] = None    # weights out without weights in
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[18] = None                     # status missing
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[17] = -1                       # negative SM count
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    # layout + dispatch: the dispatch's checks run before the layout is launched
    f2 = lib.ep_layout_and_dispatch
    f2.restype = ctypes.c_int32
    f2.argtypes = [vp, vp, vp] + [ctypes.c_int] * 7 + [ctypes.POINTER(B.ep_layout_t), vp, ctypes.c_size_t,
                                                      ctypes.c_int, ctypes.c_int64, vp, vp, ctypes.c_int, vp, vp, vp,
                                                      vp, vp]
    fargs = [vp(16), vp(32), vp(48), 10, 7168, 8, 256, 8, 0, 1, ctypes.byref(L2), vp(256), 1 << 20, B.EP_BF16, 100,
             vp(64), None, 0, None, None, None, st, None]
    bad = list(fargs); bad[4] = 7164                     # H % 8
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[13] = B.EP_FP8_E4M3           # FP8 needs recv_sf
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[15] = None                    # recv_x missing
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[0] = vp(18)                   # x misaligned
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[21] = None                    # status missing
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[7] = 4096                     # more experts than the limit
    assert f2(*bad) == B.EP_ERR_UNSUPPORTED
    bad = list(fargs); bad[10] = ctypes.byref(L4)        # layout check: src_dst_count needs R | T
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(fargs); bad[11] = None                    # workspace missing (layout check)
    assert f2(*bad) == B.EP_ERR_INVALID_ARG
    # combine
    c = lib.ep_combine
    c.restype = ctypes.c_int32
    c.argtypes = [vp, ctypes.c_int64, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.POINTER(B.ep_layout_t), vp, ctypes.c_int, vp, vp]
    cargs = [vp(16), 100, vp(32), None, 10, 7168, 8, 256, 8, ctypes.byref(L2), vp(64), 0, st, None]
    bad = list(cargs); bad[5] = 100                      # H % 8
    assert c(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(cargs); bad[10] = None                    # out missing
    assert c(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(cargs); bad[3] = vp(48); bad[2] = None    # weighted without topk_idx
    assert c(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(cargs); bad[0] = None                     # y missing with rows > 0
    assert c(*bad) == B.EP_ERR_INVALID_ARG


def _sm_rule(lib):
    f = lib.ep_theoretical_num_sms
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 6 + [ctypes.c_double] * 3 + [ctypes.c_int] * 2
    return f


def test_sm_count_rule_matches_oracle(lib):
    """The library's SM count rule against the oracle's over a grid; a case
    whose unrounded 1.25 n sits within 1e-9 of an integer may round either
    way (the two sides evaluate the binomial ratio in different orders)."""
    import itertools
    import math

    import oracle
    f = _sm_rule(lib)
    checked = 0
    for (H, K, E, R), fp8, comb, hbm, (rd, wr), ov, dev in itertools.product(
            [(7168, 8, 256, 8), (7168, 8, 256, 64), (4096, 6, 64, 16), (128, 1, 16, 4), (2048, 32, 2048, 1024),
             (256, 4, 8, 8), (1024, 8, 256, 1)],
            [False, True], [False, True], [6677.2, 1000.0, 450.0], [(200.0, 50.0), (41.0, 50.0), (10.0, 10.0)],
            [True, False], [152, 132, 16]):
        want, n = oracle.theoretical_num_sms(H, K, E, R, hbm, fp8=fp8, combine=comb, sm_read_gbs=rd,
                                             sm_write_gbs=wr, prefer_overlap=ov, device_sms=dev)
        got = f(H, K, E, R, 1 if fp8 else 0, int(comb), hbm, rd, wr, int(ov), dev)
        x = 1.25 * n
        if abs(x - round(x)) < 1e-9 * max(1.0, x):
            assert abs(got - want) <= 2
            continue
        assert got == want, (H, K, E, R, fp8, comb, hbm, rd, wr, ov, dev)
        checked += 1
    assert checked > 1000


def test_sm_count_rule_rejects_bad_arguments(lib):
    f = _sm_rule(lib)
    ok = (7168, 8, 256, 8, 0, 0, 6677.0, 200.0, 50.0, 1, 152)
    assert f(*ok) > 0
    bad = [
        (0,) + ok[1:], (100,) + ok[1:], (7176, 8, 256, 8, 1) + ok[5:],   # hidden: zero, not /8, FP8 not /128
        ok[:1] + (0,) + ok[2:], ok[:1] + (33,) + ok[2:], (7168, 8, 4, 4) + ok[4:],    # K
        ok[:3] + (7,) + ok[4:], ok[:4] + (2,) + ok[5:],                                # R does not divide E; dtype
        ok[:6] + (0.0,) + ok[7:], ok[:7] + (-1.0,) + ok[8:], ok[:8] + (float("nan"),) + ok[9:],
        ok[:10] + (0,),
    ]
    for a in bad:
        assert f(*a) == 0, a


def test_hierarchical_host_checks(lib):
    """Node rows and the two-stage calls reject bad arguments before any launch."""
    from combine_ep_get_gb300 import binding as B
    vp = ctypes.c_void_p
    st = vp(16)
    f = lib.ep_get_layout
    f.restype = ctypes.c_int32
    f.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.POINTER(B.ep_layout_t), vp, ctypes.c_size_t, vp, vp]
    fields = dict(num_tokens_per_rank=16, num_tokens_per_node=128, num_tokens_per_expert=32, is_token_in_rank=48,
                  rank_offset=64, expert_offset=80, dst_row=96, node_offset=144, node_row=160)
    ok = B.ep_layout_t(**fields)
    assert f(vp(16), 10, 8, 256, 8, 4, 1, ctypes.byref(B.ep_layout_t(**{**fields, "node_offset": None})),
             vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG          # node_row without node_offset
    assert f(vp(16), 10, 8, 256, 8, 4, 1, ctypes.byref(B.ep_layout_t(**{**fields, "node_row": None})),
             vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG          # node_offset without node_row, T > 0
    assert f(vp(16), 10, 8, 256, 8, 0, 1, ctypes.byref(ok), vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG
    assert f(vp(16), 10, 8, 256, 8, 4, 1, ctypes.byref(B.ep_layout_t(**{**fields, "num_tokens_per_node": None})),
             vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG          # no node counts
    assert f(vp(16), 10, 8, 256, 8, 4, 1, ctypes.byref(B.ep_layout_t(**{**fields, "node_row": 161})),
             vp(256), 1 << 20, st, None) == B.EP_ERR_INVALID_ARG          # misaligned
    d = lib.ep_dispatch_hierarchical
    d.restype = ctypes.c_int32
    d.argtypes = [vp, vp, vp] + [ctypes.c_int] * 6 + [ctypes.POINTER(B.ep_layout_t), ctypes.c_int, ctypes.c_int64,
                                                       vp, vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int, vp, vp, vp,
                                                       vp, vp]
    args = [vp(16), vp(32), vp(48), 10, 7168, 8, 256, 8, 4, ctypes.byref(ok), B.EP_BF16, 20, vp(64), None, None,
            100, vp(80), None, 0, None, None, None, st, None]
    bad = list(args); bad[8] = 3                                             # rpn does not divide R
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[9] = ctypes.byref(B.ep_layout_t(**{**fields, "node_row": None}))
    assert d(*bad) == B.EP_ERR_INVALID_ARG                                   # layout without node rows
    bad = list(args); bad[10] = B.EP_FP8_E4M3; bad[16] = vp(80); bad[17] = vp(96)
    assert d(*bad) == B.EP_ERR_INVALID_ARG                                   # FP8 needs node_sf
    bad = list(args); bad[12] = None                                         # node_x missing
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(args); bad[11] = -1                                           # node capacity
    assert d(*bad) == B.EP_ERR_INVALID_ARG
    c = lib.ep_combine_hierarchical
    c.restype = ctypes.c_int32
    c.argtypes = [vp, ctypes.c_int64, vp, vp] + [ctypes.c_int] * 6 + [ctypes.POINTER(B.ep_layout_t),
                                                                       ctypes.c_int64, vp, vp, vp, vp]
    cargs = [vp(16), 100, vp(32), None, 10, 7168, 8, 256, 8, 4, ctypes.byref(ok), 20, vp(48), vp(64), st, None]
    bad = list(cargs); bad[12] = None                                        # node_y missing
    assert c(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(cargs); bad[9] = 0                                            # rpn
    assert c(*bad) == B.EP_ERR_INVALID_ARG
    bad = list(cargs); bad[10] = ctypes.byref(B.ep_layout_t(**{**fields, "node_row": None}))
    assert c(*bad) == B.EP_ERR_INVALID_ARG
