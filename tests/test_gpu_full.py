"""The five workloads at full size on the GPU, checked on sampled rows against
the fp64 oracle (the oracle computes each sampled row exactly), plus the
split-count sweep of the long batch-1 decode."""
import numpy as np
import pytest
import torch

import paged_varlen_attention_causal_gb300 as ink
from test_gpu_parity import check, errors_of_last_call, gpu_run, oracle_run, sampled_rows
from workloads import workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.mark.parametrize("name,nrows", [("decode_batch", 256), ("chunked_prefill", 192), ("long_decode", 64),
                                        ("continuous_batch", 256)])
def test_workload_full_size(name, nrows):
    case = workload(name, device="cuda")
    out, lse = gpu_run(case)
    assert errors_of_last_call() & ~ink.DEVERR["EMPTY_ROWS"] == 0
    assert torch.isfinite(out.float()).all()
    rows = sampled_rows(case, nrows, 7)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    check(out, lse, ref_out, ref_lse, rows=rows, what=name)
    del case, out, lse
    torch.cuda.empty_cache()


def test_long_decode_split_sweep():
    case = workload("long_decode", device="cuda")
    rows = np.arange(case.H, dtype=np.int64)
    ref_out, ref_lse = oracle_run(case, rows=rows)
    for s in (16, 32, 64, 128):
        out, lse = gpu_run(case, num_splits=s)
        check(out, lse, ref_out, ref_lse, rows=rows, what=f"long_decode splits={s}")
    del case
    torch.cuda.empty_cache()
