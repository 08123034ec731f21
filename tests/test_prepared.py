"""cr.prepare on the CPU: what it refuses to record, and that a prepared
call is validated by the library at every invocation.  No call here carries
a device pointer, so nothing can launch."""
import pytest

from fsdp_emulated_ranks_gb300 import cr


def test_prepare_refuses_calls_with_side_effects():
    with pytest.raises(TypeError, match="cr_bucket_plan"):
        cr.prepare(cr.cr_bucket_plan, [10, 20], 2, 1024)
    with pytest.raises(ValueError, match="launches nothing"):
        cr.prepare(cr.cr_chunk_len, 10, 2)


def test_prepared_call_is_validated_at_every_invocation():
    # no ranks and no pointers: the library rejects the call before any CUDA call
    p = cr.prepare(cr.cr_all_reduce, [], 16, "bf16", "avg", [], "bf16", 0)
    assert p.name == "cr_all_reduce"
    for _ in range(2):
        with pytest.raises(cr.CRError, match="INVALID_ARG"):
            p()


def test_prepare_is_not_reentrant_and_leaves_the_library_usable():
    def nested():
        cr.prepare(cr.cr_all_reduce, [], 16, "bf16", "avg", [], "bf16", 0)
    with pytest.raises(RuntimeError, match="nested"):
        cr.prepare(lambda: (nested(), cr.cr_all_reduce([], 16, "bf16", "avg", [], "bf16", 0)))
    assert cr.cr_chunk_len(10, 4) == 3
