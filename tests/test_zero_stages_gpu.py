"""ZeRO-1 / ZeRO-2 step = the fused FSDP step.

"Distributed Training" section 4 (ZeRO-1 and ZeRO-2) gives both stages the
same per-step flow as FSDP: reduce-scatter of the gradient to the owner's
shard, the owner's optimizer update on its state shard, all-gather of the
updated parameters into full replicas; the stages differ only in how long
the reduced gradient shard is kept (ZeRO-2 keeps it as sharded state).  So
the three calls a ZeRO-2 caller makes -- cr_reduce_scatter to fp32 shards
(kept), cr_adamw_step on each shard, cr_all_gather of the bf16 shards --
must give cr_fsdp_step's parameters and optimizer state bit for bit."""
import pytest
import torch

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def filled(count, dtype, std, seed):
    t = torch.empty(count, dtype=dtype, device="cuda")
    I.torch_fill_normal_(t, std, seed)
    return t


@pytest.mark.parametrize("n,count", [(8, 8 * 8 * 4096), (8, 1_000_003), (4, 77), (3, 4097), (8, 5)])
def test_zero2_three_calls_equal_the_fused_step(n, count):
    grads = [filled(count, torch.bfloat16, 1e-3, 1000 + r) for r in range(n)]
    L = cr.cr_chunk_len(count, n)
    lens = [max(0, min(count, (j + 1) * L) - min(count, j * L)) for j in range(n)]
    master = [filled(k, torch.float32, 0.02, 2000 + j) if k else
              torch.empty(0, dtype=torch.float32, device="cuda") for j, k in enumerate(lens)]
    m = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
    v = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
    fused = ([x.clone() for x in master], [x.clone() for x in m], [x.clone() for x in v])
    zero2 = ([x.clone() for x in master], [x.clone() for x in m], [x.clone() for x in v])
    cfg = cr.adamw_cfg()

    params_fused = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    params_zero2 = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    for step in (1, 2):
        cfg.step = step
        cr.cr_fsdp_step(grads, count, *fused, cfg, params_fused)

        g_shards = [torch.empty(k, dtype=torch.float32, device="cuda") for k in lens]
        cr.cr_reduce_scatter(grads, count, "bf16", "avg", [g if g.numel() else None
                                                           for g in g_shards], "f32")
        p_shards = [torch.empty(k, dtype=torch.bfloat16, device="cuda") for k in lens]
        for j in range(n):
            if lens[j]:
                cr.cr_adamw_step(lens[j], zero2[0][j], zero2[1][j], zero2[2][j], g_shards[j],
                                 cfg, p_shards[j])
        cr.cr_all_gather([p if p.numel() else None for p in p_shards], count, "bf16",
                         params_zero2)
        torch.cuda.synchronize()
        for a, b in zip(params_fused, params_zero2):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        for part_f, part_z in zip(fused, zero2):
            for a, b in zip(part_f, part_z):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
