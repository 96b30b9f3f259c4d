"""Every hand-worked sampler case of tests/golden/sampler_cases.txt through the CUDA sampler.

The cases ("GPT-OSS Tail Chunked Megakernel Kernel API Reference", parameter
`sampling_params`; each expected token derived by hand in the file) include NaN and extreme
values of top_k, top_p, temperature and u.  tail_merge_shards takes candidate values and ids
directly: each case's sorted candidates go in as one shard, and the kernel's top-k and sampler
(the code the tail's row owners and merge kernel run) must draw the case's token.  The values
are rounded to fp32 on the way; every case keeps its order and its oracle token after that
rounding (checked below on the CPU side too).
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _golden_cases

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_sampler_case_on_the_gpu(case):
    name, vals, idx, p, want = case
    dev = torch.device("cuda:0")
    v32 = vals.astype(np.float32)
    assert oracle.sample_row(v32.astype(np.float64), idx, p).token == want  # the case survives fp32
    n = v32.size
    cv = torch.from_numpy(v32.reshape(1, 1, n)).to(dev)
    ci = torch.from_numpy(idx.astype(np.int32).reshape(1, 1, n)).to(dev)
    prm = torch.from_numpy(p.reshape(1, -1)).to(dev)
    tok = torch.full((1,), -7, dtype=torch.int32, device=dev)
    tv = torch.empty((1, n), dtype=torch.float32, device=dev)
    ti = torch.empty((1, n), dtype=torch.int32, device=dev)
    dst.merge_shards(cv, ci, [0], n, params=prm, out_tokens=tok, out_topk_vals=tv, out_topk_idx=ti)
    torch.cuda.synchronize()
    assert np.array_equal(ti.cpu().numpy()[0], idx)
    assert int(tok.cpu().numpy()[0]) == want, name
