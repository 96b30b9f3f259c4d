"""The vocabulary-parallel tail on one GPU ("simulated shards"): every slice
runs the tail with its own weight columns and no sampler, the slices' top-k
lists are merged by tail_merge_shards, and the result must equal the
unsharded tail bit for bit when both run the same lm_head realisation (the
arithmetic for a column does not depend on how the vocabulary is split) --
tokens, top-k ids and values."""
import numpy as np
import pytest

import gen
from tests import tailcheck as tc

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import decode_sampling_tail_gb300 as dst  # noqa: E402
from decode_sampling_tail_gb300.vocab_parallel import ShardedTail  # noqa: E402


@pytest.fixture(params=["gemv", "tensor"])
def path(request):
    return request.param


def unsharded(w, dev, path="auto"):
    hidden, gamma, w_t, params = dev
    with dst.Tail(w.H, w.V, w.k, w.B, hidden_actual=w.Hu, eps=w.eps, hidden_dtype=w.hidden_dtype,
                  zero_interleaved_pad=bool(w.zero_pad), path=path) as t:
        return tc.run_gpu(t, w, torch, dev_tensors=dev)


def sharded(w, dev, nshard, params_form="all", path="auto"):
    hidden, gamma, w_t, params = dev
    vals = torch.empty((nshard, w.B, w.k), dtype=torch.float32, device="cuda")
    idx = torch.empty((nshard, w.B, w.k), dtype=torch.int32, device="cuda")
    ranks = [ShardedTail(w.H, w.V, w.k, w.B, s, nshard, hidden_actual=w.Hu, eps=w.eps,
                         hidden_dtype=w.hidden_dtype, zero_interleaved_pad=bool(w.zero_pad), path=path)
             for s in range(nshard)]
    try:
        for s, rk in enumerate(ranks):
            w_slice = w_t[:, rk.lo:rk.hi].contiguous()
            rk.local_topk(hidden, gamma, w_slice, vals[s], idx[s])
        p = None if params_form == "none" else (params[:, :3].contiguous() if params_form == "3col" else params)
        tok = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        tv = torch.empty((w.B, w.k), dtype=torch.float32, device="cuda")
        ti = torch.empty((w.B, w.k), dtype=torch.int32, device="cuda")
        ranks[0].merge(vals, idx, p, tok, out_topk_vals=tv, out_topk_idx=ti)
        torch.cuda.synchronize()
        for rk in ranks:
            rk.tail.check()
        return tok.cpu().numpy(), tv.cpu().numpy(), ti.cpu().numpy()
    finally:
        for rk in ranks:
            rk.close()


@pytest.mark.parametrize("nshard", [2, 8])
def test_gptoss_g8_vocab_shards_equal_the_unsharded_tail(nshard, path):
    w = gen.make("gptoss_g8")
    dev = tc.to_device(w, torch)
    ref = unsharded(w, dev, path)
    tok, tv, ti = sharded(w, dev, nshard, path=path)
    assert np.array_equal(ti, ref.topk_idx)
    assert np.array_equal(tv.view(np.uint32), ref.topk_vals.view(np.uint32))
    assert np.array_equal(tok, ref.tokens)


@pytest.mark.parametrize("shape", [(5, 128, 4096, 64, "f16"), (20, 160, 8192, 100, "bf16"), (70, 64, 6144, 33, "f32")],
                         ids=lambda s: f"B{s[0]}_V{s[2]}_k{s[3]}")
def test_small_vocab_shards_equal_the_unsharded_tail_and_the_oracle(shape, path):
    B, H, V, k, dt = shape
    w = gen.custom(B, H, V, k, hidden_dtype=dt, seed=4000 + B, dup_cols=2)  # ties that straddle slice edges
    dev = tc.to_device(w, torch)
    ref = unsharded(w, dev, path)
    tok, tv, ti = sharded(w, dev, 3, path=path)
    assert np.array_equal(ti, ref.topk_idx) and np.array_equal(tok, ref.tokens)
    L, ov, oi = tc.oracle_rows(w, np.arange(B))
    tc.check_topk(tv, ti, L, ov, oi, w.k, ref.logits)


def test_merge_without_sampler_leaves_tokens_and_rejects_bad_arguments():
    w = gen.custom(4, 64, 2048, 16, hidden_dtype="bf16", seed=4100)
    dev = tc.to_device(w, torch)
    tok, tv, ti = sharded(w, dev, 2, params_form="none")
    assert np.all(tok == -7)
    ref = unsharded(w, dev)
    assert np.array_equal(ti, ref.topk_idx)
    tok3, _, _ = sharded(w, dev, 2, params_form="3col")
    assert tok3.shape == (4,)
    v = torch.zeros((2, 4, 16), device="cuda")
    i = torch.zeros((2, 4, 16), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert dst.tail_merge_shards(2, 16, 33, 4, v.data_ptr(), i.data_ptr(), [0, 1024], None, 4, None, None, None,
                                 s) == dst.TAIL_ERR_INVALID_ARG  # k above nshard * k_in
    assert dst.tail_merge_shards(0, 16, 8, 4, v.data_ptr(), i.data_ptr(), [], None, 4, None, None, None,
                                 s) == dst.TAIL_ERR_INVALID_ARG


@pytest.mark.parametrize("nshard", [2, 4])
def test_owned_row_blocks_draw_the_unsharded_tokens(nshard, path):
    # the all-to-all of owned rows, simulated: rank q merges [nshard, gbs / nshard, k] candidates of
    # its row block with only its rows' sampling parameters
    from decode_sampling_tail_gb300.vocab_parallel import owned_row_block
    w = gen.custom(8, 256, 16384, 64, hidden_dtype="bf16", seed=4200, dup_cols=2)
    dev = tc.to_device(w, torch)
    hidden, gamma, w_t, params = dev
    ref = unsharded(w, dev, path)
    vals = torch.empty((nshard, w.B, w.k), dtype=torch.float32, device="cuda")
    idx = torch.empty((nshard, w.B, w.k), dtype=torch.int32, device="cuda")
    ranks = [ShardedTail(w.H, w.V, w.k, w.B, s, nshard, path=path) for s in range(nshard)]
    try:
        for s, rk in enumerate(ranks):
            rk.local_topk(hidden, gamma, w_t[:, rk.lo:rk.hi].contiguous(), vals[s], idx[s])
        for q, rk in enumerate(ranks):
            r0, n = owned_row_block(q, nshard, w.B)
            tok = torch.full((n,), -7, dtype=torch.int32, device="cuda")
            ti = torch.empty((n, w.k), dtype=torch.int32, device="cuda")
            rk.merge(vals[:, r0:r0 + n].contiguous(), idx[:, r0:r0 + n].contiguous(),
                     params[r0:r0 + n].contiguous(), tok, out_topk_idx=ti)
            torch.cuda.synchronize()
            assert np.array_equal(tok.cpu().numpy(), ref.tokens[r0:r0 + n])
            assert np.array_equal(ti.cpu().numpy(), ref.topk_idx[r0:r0 + n])
    finally:
        for rk in ranks:
            rk.close()
