"""ra_bwd_noalloc: the backward for callers that cannot allocate device memory
(for instance a plugin whose host framework owns all device memory, or a code
path that must not call cudaMalloc because it can synchronise the device).

It must give exactly what ra_bwd gives with a caller-allocated workspace,
call after call, while allocating nothing.  The backward kernels are
deterministic (every output row has one writer and no atomics), so the check is
bit equality: a stale value left in the shared array by an earlier call would
show up as a difference in even one row.  This file is collected last on purpose, so a
run that stops at the first failure has run every other test first; it also
passes on its own in a fresh process.
"""
import pytest
import torch

from ring_attention_fwd_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_no_alloc_backward_matches_workspace_backward():
    import ring_attention_fwd_gb300 as ra
    L = ra.binding.lib()
    B, H, S, D, N = 1, 4, 2048, 128, 4
    for causal, layout in ((True, "striped"), (True, "contiguous")):
        x = {k: v.cuda() for k, v in make_inputs(B, H, S, D, seed=77, with_grad=True).items()}
        o, lse = ra.fwd(x["q"], x["k"], x["v"], N, causal, layout)
        ref = ra.bwd(x["q"], x["k"], x["v"], o, lse, x["do"], N, causal, layout)
        outs = [torch.empty_like(x["q"]) for _ in range(3)]
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):          # two calls in a row share the library's array
            for t in outs:
                t.fill_(float("nan"))
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            rc = L.ra_bwd_noalloc(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), x["do"].data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(),
                                  outs[2].data_ptr(), B, H, S, D, N, int(causal), ra.binding._LAYOUT[layout],
                                  ra.binding.RA_BF16, stream)
            assert rc == 0, L.ra_last_error().decode()
            torch.cuda.synchronize()
            ra.check_device_status()
            if call == 1:              # the first call may load the library's module; later ones change nothing
                assert torch.cuda.mem_get_info()[0] == free_before
            for name, g, r in zip(("dQ", "dK", "dV"), outs, ref):
                assert torch.equal(g, r), f"{name} (call {call}, {layout}) differs from ra_bwd"


def test_no_alloc_backward_rejects_too_large():
    import ring_attention_fwd_gb300 as ra
    x = torch.empty((1, 64, 131072, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 64, 131072), dtype=torch.float32, device="cuda")
    with pytest.raises(ra.RingAttnError, match="more than the fixed"):
        ra.bwd_noalloc(x, x, x, x, lse, x, 32, True, "contiguous", dq=x, dk=x, dv=x)
