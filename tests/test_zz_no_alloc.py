"""The clipped FSDP step for callers that cannot allocate device memory.

cr_fsdp_step_clipped_noalloc keeps its scratch in the library's own static
device array, for callers (framework plugins handed only their tensors,
code that must not trigger a synchronising cudaMalloc) that have no
workspace to pass.  Called through the C ABI, it must give what
cr_fsdp_step_clipped gives with a caller workspace, on two calls in a row
(the second starting from the state the first left, and reusing the static
array the first call filled), and both calls must equal the oracle's clipped
step bit for bit at a clip coefficient the oracle's norm allows.  This file
is collected last on purpose.
"""
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_clipped_match, assert_match, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def make_state(n, count, L):
    master_full = torch.empty(count, dtype=torch.float32, device="cuda")
    I.torch_fill_normal_(master_full, 0.02, 2000)
    master = [master_full[j * L:min((j + 1) * L, count)].clone() for j in range(n)]
    m = [torch.zeros_like(x) for x in master]
    v = [torch.zeros_like(x) for x in master]
    params = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    return master, m, v, params


@pytest.mark.parametrize("n,count,max_norm", [(8, 8 * 8 * 4096 + 5, 1e-3), (4, 100003, 1e30)])
def test_noalloc_matches_workspace_call_twice(n, count, max_norm):
    L = cr.cr_chunk_len(count, n)
    ws_bytes = cr.cr_fsdp_clip_workspace_bytes()
    ws = torch.empty(ws_bytes // 8, dtype=torch.float64, device="cuda")
    a_state = make_state(n, count, L)   # caller-workspace entry point
    b_state = make_state(n, count, L)   # static-scratch entry point
    a_norm = torch.empty(1, dtype=torch.float32, device="cuda")
    b_norm = torch.empty(1, dtype=torch.float32, device="cuda")
    # The oracle's copy of the state, advanced alongside the GPU's.
    h_state = [[to_host(x, "f32") for x in t] for t in b_state[:3]]
    for step in (1, 2):
        grads = []
        for r in range(n):
            g = torch.empty(count, dtype=torch.bfloat16, device="cuda")
            I.torch_fill_normal_(g, 1e-3, 1000 + 31 * step + r)
            grads.append(g)
        cfg = cr.adamw_cfg(step=step)
        am, amm, av, ap = a_state
        bm, bmm, bv, bp = b_state
        cr.cr_fsdp_step_clipped(grads, count, am, amm, av, cfg, max_norm, ws, ws_bytes, ap, a_norm)
        cr.cr_fsdp_step_clipped_noalloc(grads, count, bm, bmm, bv, cfg, max_norm, bp, b_norm)
        torch.cuda.synchronize()
        # Same kernels, same first-pass grid, same fixed summation order:
        # the two entry points agree bit for bit, norm included.
        assert_match(to_host(b_norm, "f32"), to_host(a_norm, "f32"), "f32", f"norm, step {step}")
        for x, y in zip(am + amm + av, bm + bmm + bv):
            assert_match(to_host(y, "f32"), to_host(x, "f32"), "f32", f"state, step {step}")
        for x, y in zip(ap, bp):
            assert_match(to_host(y, "bf16"), to_host(x, "bf16"), "bf16", f"params, step {step}")
        # And against the oracle: the norm to its summation-order tolerance,
        # everything after the coefficient bitwise.
        h_grads = [to_host(g, "bf16") for g in grads]
        ocfg = O.AdamWConfig(step=step)
        _, want_norm = O.fsdp_step_clipped(h_grads, [x.copy() for x in h_state[0]],
                                           [x.copy() for x in h_state[1]],
                                           [x.copy() for x in h_state[2]], ocfg, max_norm)
        assert float(b_norm.item()) == pytest.approx(want_norm, rel=1e-6)
        got_state = [[to_host(x, "f32") for x in t] for t in (bm, bmm, bv)]
        assert_clipped_match(got_state, [to_host(x, "bf16") for x in bp], h_grads, *h_state,
                             ocfg, max_norm, want_norm, f"step {step}")


def test_noalloc_rejects_bad_arguments_before_launch():
    with pytest.raises(cr.CRError) as ei:
        cr.cr_fsdp_step_clipped_noalloc([0] * 2, 16, [0] * 2, [0] * 2, [0] * 2, cr.adamw_cfg(),
                                        1.0, [0] * 2)
    assert ei.value.status == 1
