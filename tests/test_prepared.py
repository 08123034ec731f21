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


def test_every_stream_entry_point_is_preparable_unless_it_keeps_host_state():
    """Every entry point of the C ABI that enqueues work on a stream can be
    prepared, except those whose host-side state a replay would corrupt:
    the reducer's and communicator's, which track calls between invocations,
    and the checked build's self-test."""
    import os
    import re
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "include", "cr.h")
    decls = re.findall(r"\bcr_status\s+(cr_\w+)\s*\(([^;]*?)\);", open(header).read(), re.S)
    streamed = {name for name, params in decls if "cr_stream_t" in params}
    stateful = {"cr_reducer_create", "cr_reducer_mark_ready", "cr_reducer_finalize",
                "cr_comm_create", "cr_check_selftest"}
    assert len(streamed) > 20
    assert sorted(streamed - stateful - cr._PREPARABLE) == []
    assert not (stateful & cr._PREPARABLE)


def test_a_prepared_slab_split_may_compute_its_slabs_while_recording():
    # host-only helpers run for real while prepare() records; the range calls
    # are recorded (and rejected at invocation: no ranks, no pointers)
    def split():
        for g in range(3):
            lo, hi = cr.cr_slab_range(1000, 4, 3, g)
            cr.cr_all_reduce_range([], 1000, lo, hi, "bf16", "avg", [], "bf16", 0)
    p = cr.prepare(split)
    assert len(p._calls) == 3 and {c[0] for c in p._calls} == {"cr_all_reduce_range"}
    with pytest.raises(cr.CRError, match="INVALID_ARG"):
        p()
