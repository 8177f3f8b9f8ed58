"""The allocation-free decode entry point, cpe_decode_attention_noalloc.

Some callers cannot allocate device memory at all: a plugin running inside a
host program that owns every byte of device memory through its own pool, or a
serving loop that must not enter an allocator on its hot path (cudaMalloc can
synchronise the device, and can fail on a fragmented heap).  For them the
split-KV decode path keeps its partial results in a fixed 8 MiB device array
that the library declares itself, instead of a workspace the caller would have
to allocate.

These tests call that entry point through the C ABI and check it against the
float64 oracle and against the workspace-based cpe_decode_attention, twice in
a row (the fixed array is shared by every call and keeps the previous call's
contents); that a call after the first leaves the device's free memory where
it was, and that each call launches only the decode kernels; and that a batch needing more than the fixed
array is refused before anything is launched.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._util import MAX_ABS, REL_RMS, LSE_ABS, check_close, i32, varlen_batch


def _lib():
    from chunked_prefill_extend_gb300 import cpe
    return cpe


def _both_paths(cpe, b):
    """Append the new rows, then run the workspace path and the fixed-array path.
    Returns both results and, for the fixed-array call, the device's free bytes
    before and after it and the kernels it launched."""
    pl = i32(b["pl"])
    cpe.cpe_kv_append(b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["page_table"], i32(b["qo"]), pl)
    n, h_q = b["q"].shape[0], b["h_q"]
    lse_ref = torch.empty(n, h_q, dtype=torch.float32, device="cuda")
    ref, _ = cpe.cpe_decode_attention(b["q"], b["k_cache"], b["v_cache"], b["page_table"], pl, b["max_kv"],
                                      lse=lse_ref)
    out = torch.empty_like(b["q"])
    lse = torch.empty(n, h_q, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    launches0 = cpe.cpe_launch_count()
    cpe.cpe_decode_attention_noalloc(b["q"], b["k_cache"], b["v_cache"], b["page_table"], pl, b["max_kv"],
                                     out=out, lse=lse)
    launched = cpe.cpe_launch_count() - launches0
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    st, detail = cpe.cpe_get_device_status()
    assert st == cpe.CPE_OK, f"device status {st} ({detail})"
    return out, lse, ref, lse_ref, free0, free1, launched


@pytest.mark.gpu
def test_noalloc_decode_matches_oracle_and_workspace_path_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cpe = _lib()
    # first call: several splits per row; second call: other rows, other sizes
    first = varlen_batch(901, [(L - 1, 1) for L in (1, 17, 2049, 6000, 9000)], 32, 8, 128)
    second = varlen_batch(902, [(L - 1, 1) for L in (4097, 33, 12000)], 16, 4, 64)
    for k, b in enumerate((first, second)):
        out, lse, ref, lse_ref, free0, free1, launched = _both_paths(cpe, b)
        # the float64 oracle on the appended cache (a decode row is an extend row at P = L - 1)
        ref_o, ref_l = oracle.extend_attention(b["q"].cpu(), b["k_cache"].cpu(), b["v_cache"].cpu(),
                                               b["page_table_host"], b["qo"], b["pl"], b["h_q"], b["h_kv"])
        check_close(out, ref_o, "noalloc vs oracle")
        np.testing.assert_allclose(lse.cpu().numpy(), ref_l, atol=LSE_ABS, rtol=0)
        check_close(out, ref.double().cpu().numpy(), "noalloc vs workspace path", MAX_ABS, REL_RMS)
        np.testing.assert_allclose(lse.cpu().numpy(), lse_ref.cpu().numpy(), atol=LSE_ABS, rtol=0)
        # The first call in a process may load the library's device module (CUDA
        # loads modules lazily), which places the fixed array on the device; from
        # then on a call takes no device memory.
        if k > 0:
            assert free1 == free0, f"device free memory moved by {free0 - free1} bytes across the call"
        assert launched in (1, 2), launched  # the decode kernel, and the merge of splits when there are several


def test_noalloc_refuses_batches_above_the_fixed_array():
    """64 rows x 32 heads x 16 splits x 130 floats needs ~17 MB > 8 MiB: refused on
    the host with CPE_ERR_CAPACITY, before any device call (the pointers are
    never dereferenced)."""
    cpe = _lib()
    fake = 1 << 20
    st = cpe._lib.cpe_decode_attention_noalloc(fake, fake, fake, 100000, fake, 2048, fake, 64, 32768, 32, 8, 128,
                                                16, 0.088, cpe.CPE_BF16, fake, None, None)
    assert st == cpe.CPE_ERR_CAPACITY
    assert "8388608" in cpe.cpe_last_error()
