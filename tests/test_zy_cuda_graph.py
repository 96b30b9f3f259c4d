"""The tail captured in a CUDA graph and replayed.

A run is asynchronous on the caller's stream and makes no host synchronisation, so steps can be
captured once and replayed.  Each replay must give the outputs of an eager run bit for bit: the
per-row arrival words between CTAs reset themselves at the end of every run, and the tensor maps
travel by value in the kernel parameters, so nothing needs a host-side reset between replays.
Two captured steps read two input buffers whose contents change between replays.
"""
import dataclasses

import numpy as np
import pytest

import gen
from tests import tailcheck as tc
from tests.test_gpu_parity import make_tail

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)


def _outputs(B, V, k, dev):
    return (torch.full((B,), -7, dtype=torch.int32, device=dev), torch.empty((B, V), dtype=torch.float32, device=dev),
            torch.empty((B, k), dtype=torch.float32, device=dev), torch.empty((B, k), dtype=torch.int32, device=dev))


def _same(out, ref):
    tokens, logits, tv, ti = (x.cpu().numpy() for x in out)
    assert np.array_equal(logits.view(np.uint32), ref.logits.view(np.uint32))
    assert np.array_equal(tv.view(np.uint32), ref.topk_vals.view(np.uint32))
    assert np.array_equal(ti, ref.topk_idx)
    assert np.array_equal(tokens, ref.tokens)


@pytest.mark.parametrize("path", ["gemv", "tensor", "small"])
def test_graph_replays_match_eager_runs(path):
    dev = torch.device("cuda:0")
    w1 = gen.custom(8, 512, 16384, 64, hidden_dtype="bf16", seed=401)
    w2 = dataclasses.replace(w1, hidden=gen.custom(8, 512, 16384, 64, hidden_dtype="bf16", seed=402).hidden)
    with make_tail(w1, path=path) as t:
        hid1, gamma, w_t, p = tc.to_device(w1, torch)
        hid2 = tc.to_device(w2, torch)[0]
        r1 = tc.run_gpu(t, w1, torch, dev_tensors=(hid1, gamma, w_t, p))
        r2 = tc.run_gpu(t, w2, torch, dev_tensors=(hid2, gamma, w_t, p))

        in_a, in_b = torch.empty_like(hid1), torch.empty_like(hid1)
        out_a, out_b = _outputs(w1.B, w1.V, w1.k, dev), _outputs(w1.B, w1.V, w1.k, dev)

        def step():
            for x, (tok, lg, tv, ti) in ((in_a, out_a), (in_b, out_b)):
                t.run(x, gamma, w_t, p, out_tokens=tok, out_logits=lg, out_topk_vals=tv, out_topk_idx=ti)

        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            in_a.copy_(hid1)
            in_b.copy_(hid2)
            step()  # warm state on the capture stream
        torch.cuda.synchronize(dev)
        t.check()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for first, second in ((hid1, hid2), (hid2, hid1), (hid1, hid2)):
            for o in (out_a, out_b):
                o[0].fill_(-7)
                o[1].fill_(float("nan"))
            in_a.copy_(first)
            in_b.copy_(second)
            torch.cuda.synchronize(dev)
            g.replay()
            torch.cuda.synchronize(dev)
            t.check()
            _same(out_a, r1 if first is hid1 else r2)
            _same(out_b, r2 if second is hid2 else r1)
