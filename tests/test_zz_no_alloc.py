"""dt_topm_static, the allocation-free top-M, against dt_topm (collected last on purpose).

Some callers cannot call cudaMalloc (a backend or plugin whose host framework owns all device memory, or a path that
cannot take an allocation's implicit device synchronisation); dt_topm_static serves them from one library-wide
device array. These checks call it through the C ABI directly, twice in a row with different inputs and shapes, and
require results bit-identical to dt_topm's (top-M is integer work: the tolerance is zero).
"""
import ctypes

import pytest
import torch

from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu


def _call_static(dtlib, logits, M):
    B, K, V = logits.shape
    ids = torch.full((B, K, M), -1, dtype=torch.int32, device="cuda")
    vals = torch.full((B, K, M), float("nan"), dtype=torch.float32, device="cuda")
    code = 1 if logits.dtype == torch.bfloat16 else 0
    st = dtlib.lib().dt_topm_static(logits.data_ptr(), code, B, K, V, M, ids.data_ptr(), vals.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    return st, ids, vals


def test_static_topm_matches_workspace_topm(dtlib):
    cases = [(synth.make_logits(1, device="cuda"), 64),                     # one request, 19 chunks per row
             (synth.make_logits(0, device="cuda"), 8),                      # fp32, one chunk per row
             (synth.make_logits(2, device="cuda", B=8), 64),                # 128 rows: a larger share of the array
             (synth.make_logits(4, device="cuda", B=2), 128)]
    for logits, M in cases + cases[:1]:                                     # consecutive calls, then a repeat
        ref_ids, ref_vals = dtlib.dt_topm(logits, M)
        st, ids, vals = _call_static(dtlib, logits, M)
        assert st == 0, dtlib.lib().dt_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert torch.equal(vals, ref_vals)
    # the Python binding of the same entry point (argument marshalling only)
    logits, M = cases[0]
    ids, vals = dtlib.dt_topm_static(logits, M)
    ref_ids, ref_vals = dtlib.dt_topm(logits, M)
    torch.cuda.synchronize()
    assert torch.equal(ids, ref_ids) and torch.equal(vals, ref_vals)


def test_static_topm_rejects_sizes_beyond_its_array(dtlib):
    B, K, V, M = 256, 16, 151936, 128   # 4096 rows: above the array's 1630 rows of bf16 logits at M = 128
    fake = 1 << 20                      # never dereferenced: the size check comes before any launch
    st = dtlib.lib().dt_topm_static(fake, 1, B, K, V, M, fake, fake, None)
    assert st == 2   # DT_ERR_UNSUPPORTED
