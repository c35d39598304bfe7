"""The debug build's store checks (libkvq built with -DKVQ_DEBUG=1, e.g.
KVQ_NVCC_FLAGS=-DKVQ_DEBUG=1 python -m pytest tests -m gpu): with no GPU or
memory checker on this pool, every kernel store is checked against the span
of the buffer its arguments describe, and the canary bands of
tests/_helpers.guarded catch what a check would miss.  This file shows the
checks are live in a debug build and absent from a release build."""
import pytest
import torch

from _helpers import guarded, kvq


def test_debug_entry_points_are_exported():
    K = kvq()
    assert K.kvq_debug_build() in (True, False)


@pytest.mark.gpu
def test_bounds_selftest_flags_and_skips_a_stray_store():
    """A store one byte past a one-byte span inside the pool header: a debug
    build skips it and sets KVQ_DEVERR_BOUNDS; a release build has no checks
    and refuses the self-test."""
    K = kvq()
    cfg = K.make_config(4, 16, 2, 128, "int8_per_token_head", torch.float16)
    pool = guarded(K.kvq_cache_bytes(cfg), torch.uint8, fill=0, name="pool")
    cache = K.kvq_cache_alloc(cfg, pool)
    before = pool[:256].clone()
    if not K.kvq_debug_build():
        with pytest.raises(K.KVQError) as e:
            K.kvq_debug_bounds_selftest(cache)
        assert e.value.status == 2
        return
    K.kvq_debug_bounds_selftest(cache)
    torch.cuda.synchronize()
    assert K.kvq_cache_read_errors(cache) == 0x40
    after = pool[:256]
    after[12:16] = before[12:16]          # the error word itself
    assert torch.equal(after, before)     # byte 41 was not written
