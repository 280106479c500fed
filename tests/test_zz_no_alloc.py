"""pkv_decode_noalloc: decode for callers that cannot allocate device memory
(for example a plugin whose host runtime owns all device memory, or a service
with a device-memory budget fixed at start-up).  Its scratch is an array
inside the library, shared by every call.

The test calls it through the C ABI twice in a row, on different batches.  Both
entry points run the same deterministic kernels on the same inputs, so each
output must equal pkv_decode's (the caller-workspace entry point) bit for bit;
it is also checked against the oracle within the attention tolerance the
other tests use.  A stale value left in the shared scratch by the first call
would show up as a difference in the second.  It runs last so that a failure
here leaves every other test already run, and passes both alone in a fresh
process and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from pkv_testutil import GpuBatch, assert_attention_close, bits, expect_no_device_error

pytestmark = pytest.mark.gpu


def _noalloc_via_abi(pkv, b: GpuBatch, out: torch.Tensor) -> int:
    wl = b.wl
    lib = pkv.load()
    return lib.pkv_decode_noalloc(
        ctypes.c_void_p(b.q.data_ptr()), ctypes.c_void_p(b.k_cache.data_ptr()), ctypes.c_void_p(b.v_cache.data_ptr()),
        ctypes.c_void_p(b.block_tables.data_ptr()), wl.max_blocks_per_seq, ctypes.c_void_p(b.kv_lens.data_ptr()),
        wl.batch, int(wl.kv_lens.max()), wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks,
        float(wl.softmax_scale), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_decode_on_two_calls(pkv):
    cases = [W.decode_b64(), W.decode_b64(seed=77, batch=16, lo=1, hi=700)]
    for wl in cases:                       # two calls in a row; the second sees the first's scratch contents
        b = GpuBatch(wl, W.paged_values(wl))
        b.run_slots_and_store(pkv, decode=True)
        ref = b.run_decode(pkv).clone()
        out = torch.full_like(b.q, float("nan"))
        assert _noalloc_via_abi(pkv, b, out) == 0
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(ref)), f"noalloc differs from the workspace decode ({wl.name})"
        rows = list(range(0, wl.batch, max(1, wl.batch // 16)))
        assert_attention_close(out[rows], b.oracle_decode(rows=rows), f"noalloc vs oracle ({wl.name})")
    expect_no_device_error(pkv)


def test_noalloc_rejects_batch_beyond_scratch(pkv):
    """A batch whose scratch need exceeds the built-in array is refused before any launch."""
    B = 1024
    q = torch.zeros(B, 16, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(2, 256, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(B, 1, dtype=torch.int32, device="cuda")
    ctx = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    assert pkv.pkv_decode_workspace_size(B, 16, 8, 128) > 4 * 1024 * 1024
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_noalloc(q, pool, pool, bt, ctx, 1, 0.1, out)
    assert e.value.status == 2                        # PKV_ERR_UNSUPPORTED
