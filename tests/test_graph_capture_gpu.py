"""Every entry point is asynchronous on the caller's stream and allocates no
device memory, so a whole step can be captured in a CUDA graph and replayed.
Replays must reproduce the eager results bit for bit."""
import pytest
import torch

from ring_attention_fwd_gb300.inputs import make_decode_inputs, make_ffn_inputs, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attention_fwd_gb300 as ra
    assert torch.cuda.is_available()
    return ra


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # first call outside capture: one-time attribute setup
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_fwd_bwd_step_replays_bit_exact(ra):
    B, H, S, D, N = 1, 4, 2048, 128, 4
    dev = {k: v.cuda() for k, v in make_inputs(B, H, S, D, seed=71, with_grad=True).items()}
    o = torch.empty_like(dev["q"])
    lse = torch.empty(B, H, S, device="cuda")
    dq, dk, dv = (torch.empty_like(dev["q"]) for _ in range(3))
    work = torch.empty(ra.bwd_workspace_bytes(B, H, S, D, N), dtype=torch.uint8, device="cuda")

    def step():
        ra.fwd(dev["q"], dev["k"], dev["v"], N, True, "striped", o=o, lse=lse)
        ra.bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], N, True, "striped", dq=dq, dk=dk, dv=dv,
               workspace=work)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = _capture(step)
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    ra.check_device_status()
    for a, b in zip(eager, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b)


def test_decode_and_ffn_replay_bit_exact(ra):
    dinp = {k: v.cuda() for k, v in make_decode_inputs(2, 4, 5000, 128, seed=72).items()}
    o = torch.empty_like(dinp["q"])
    lse = torch.empty(2, 4, device="cuda")
    dwork = torch.empty(ra.decode_workspace_bytes(2, 4, 5000, 128, 4), dtype=torch.uint8, device="cuda")
    finp = {k: v.cuda() for k, v in make_ffn_inputs(512, 256, 384, seed=73).items()}
    y = torch.empty_like(finp["x"])
    fwork = torch.empty(ra.ffn_workspace_bytes(512, 256, 384, 256), dtype=torch.uint8, device="cuda")

    def step():
        ra.decode(dinp["q"], dinp["k"], dinp["v"], 4, o=o, lse=lse, workspace=dwork)
        ra.ffn(finp["x"], finp["w1"], finp["w3"], finp["w2"], 256, y=y, workspace=fwork)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, y)]
    g = _capture(step)
    for t in (o, lse, y):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    ra.check_device_status()
    for a, b in zip(eager, (o, lse, y)):
        assert torch.equal(a, b)
