"""EP_GET_DEBUG: host-side logging of the C ABI (one stderr line per call,
per rejecting argument check and per kernel launch), the counterpart of the
"DeepEP Symmetric Memory" EP_BUFFER_DEBUG switch (App. B, environment
variables).  Each case runs in a child process, since the library reads the
variable once."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REJECTED = textwrap.dedent("""
    import ctypes
    from combine_ep_get_gb300 import build
    lib = ctypes.CDLL(build.build())
    from combine_ep_get_gb300 import binding as B
    L = B.ep_layout_t()
    vp = ctypes.c_void_p
    # R = 7 does not divide E = 256: rejected on the host, nothing launched
    code = lib.ep_get_layout(None, 10, 8, 256, 7, 0, 1, ctypes.byref(L), None, ctypes.c_size_t(0), vp(16), None)
    print("code", code)
""")


def _run(code, debug):
    env = dict(os.environ)
    env.pop("EP_GET_DEBUG", None)
    if debug is not None:
        env["EP_GET_DEBUG"] = debug
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_rejected_call_is_logged_with_its_check():
    r = _run(REJECTED, "1")
    assert r.returncode == 0, r.stderr
    assert "code 1" in r.stdout                      # EP_ERR_INVALID_ARG
    lines = [l for l in r.stderr.splitlines() if l.startswith("[ep_get]")]
    assert any("ep_get_layout: T=10 K=8 E=256 R=7" in l for l in lines), lines
    assert any("invalid_arg (api.cu:" in l for l in lines), lines


@pytest.mark.parametrize("value", [None, "0"])
def test_silent_unless_asked(value):
    r = _run(REJECTED, value)
    assert r.returncode == 0, r.stderr
    assert "code 1" in r.stdout
    assert "[ep_get]" not in r.stderr


STEP = textwrap.dedent("""
    import numpy as np, torch
    from combine_ep_get_gb300 import build
    build.build()
    from combine_ep_get_gb300 import binding as B
    from combine_ep_get_gb300.inputs import make_inputs
    T, H, E, K, R = 64, 1024, 64, 4, 8
    d = make_inputs(T, H, E, K, R, seed=3)
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    w = torch.from_numpy(d["topk_weights"]).cuda()
    x = torch.from_numpy(d["x_bits"].view(np.int16)).view(torch.bfloat16).cuda()
    lay = B.alloc_layout(T, E, R, 0)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, 0), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ep_get_layout(idx, E, R, lay, ws, st)
    n = lay.num_recv
    rx = torch.empty((n, H), dtype=torch.bfloat16, device="cuda")
    B.ep_dispatch(x, idx, w, E, R, lay, rx, None, None, None, st)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    B.ep_combine(rx, idx, w, E, R, lay, out, st)
    torch.cuda.synchronize()
    print("status", int(st.item()))
""")


@pytest.mark.gpu
def test_launches_are_logged():
    r = _run(STEP, "1")
    assert r.returncode == 0, r.stderr
    assert "status 0" in r.stdout
    lines = [l for l in r.stderr.splitlines() if l.startswith("[ep_get]")]
    for call in ("ep_get_layout: T=64", "ep_dispatch: T=64 H=1024", "ep_combine: T=64 H=1024"):
        assert any(call in l for l in lines), (call, lines)
    launches = [l for l in lines if " launch " in l or l.startswith("[ep_get] launch")]
    assert any("layout" in l for l in launches), launches
    assert any("dispatch_bf16_regs_kernel" in l for l in launches), launches
    assert any("combine_kernel" in l and "grid (" in l for l in launches), launches
