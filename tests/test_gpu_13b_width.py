"""Whole iterations at the 13B width (H=5120, 40 heads of 128, FFN 20480,
vocab 50257) against the oracle, on a 2-layer slice of the model.

The batches have the shapes of the two fixed 13B workloads, scaled so that
the oracle (float64, one request and one token at a time) can follow the
sampled requests:
* prefill-heavy mixed: 16 requests prefill contexts of up to 2048 tokens
  (iteration 0, ~16k rows), then two new prompts of 1024-2048 tokens run
  next to the 16 decode rows (iteration 1, the mixed shape), then decodes;
* decode-dominated: 62 requests with 1024-4096 cached tokens and two short
  ones decode together;
* a few hundred decode rows (200 short requests), where each Linear takes a
  different GEMM plan.
The integer record of every iteration (batch, rows, cached lengths, slots,
releases, K/V usage) is compared in full with the oracle scheduler; the
logits of the sampled requests (the short decodes and the shorter new
prompt) at every generated step are compared with the oracle's, under
teacher forcing (CS349D Lecture 2, section 4: batched generation equals
generating each request alone)."""
import numpy as np
import pytest

import synth
from oracle import model as omodel

from . import _harness as hz

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
SHAPE = synth.with_layers(synth.GPT_13B, 2)


@pytest.fixture(scope="module")
def cuda(liborca):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def model(cuda):
    """(host weights, oracle) of the 2-layer 13B-width slice; non-zero biases
    and LayerNorm parameters so that a dropped term shows."""
    w = synth.make_weights(SHAPE, seed=31, bias_std=0.02, ln_std=0.1)
    return w, omodel.GPTOracle(SHAPE, w)


def _req(rng, rid, arrival, n_prompt, out_len):
    return synth.Request(rid, arrival, rng.integers(0, SHAPE.vocab, n_prompt).astype(np.int32), out_len,
                         n_prompt + out_len + 2, forced=rng.integers(0, SHAPE.vocab, out_len).astype(np.int32))


def _check(model, trace, sample, max_bs, n_slots, max_rows):
    w, orc = model
    recs, eng, _ = hz.run_gpu(SHAPE, w, trace, max_bs=max_bs, n_slots=n_slots, max_rows=max_rows,
                              teacher_force=True, keep_ids={r.req_id for r in sample})
    try:
        hz.compare_schedule(recs, trace, max_bs=max_bs, n_slots=n_slots)
        got = hz.gpu_logits_by_request(recs)
        worst = 0.0
        for req in sample:
            _, logits, _ = orc.generate(req.prompt, req.out_len, forced=req.forced)
            assert len(got[req.req_id]) == req.out_len
            for k, (g, o) in enumerate(zip(got[req.req_id], logits)):
                err = hz.max_rel_err(g, o)
                worst = max(worst, err)
                assert err < BF16_TOL, (req.req_id, k, err)
        return recs, worst
    finally:
        eng.close()


def test_13b_width_prefill_heavy_mixed_iteration(cuda, model):
    rng = np.random.default_rng(32)
    # 16 requests whose prompts become the decode contexts (two short ones sampled)
    ctx = [130, 211] + rng.integers(128, 2049, 14).tolist()
    trace = [_req(rng, i, 0, int(c), 3) for i, c in enumerate(ctx)]
    # two new prompts arrive at iteration 1 (the shorter one sampled)
    trace += [_req(rng, 16, 1, 1031, 2), _req(rng, 17, 1, int(rng.integers(1024, 2049)), 2)]
    n_slots = sum(r.max_tokens for r in trace) + 64
    recs, worst = _check(model, trace, [trace[0], trace[1], trace[16]], max_bs=32, n_slots=n_slots,
                         max_rows=sum(ctx) + 64)
    # iteration 1 is the mixed shape: 16 decode rows and two prompts of >= 1024 rows
    assert sorted(recs[1].n_new) == [1] * 16 + sorted([trace[16].n_prompt, trace[17].n_prompt])
    assert sum(recs[0].n_new) == sum(ctx)


def test_13b_width_decode_dominated_iteration(cuda, model):
    rng = np.random.default_rng(33)
    ctx = [177, 302] + rng.integers(1024, 4097, 62).tolist()
    trace = [_req(rng, i, 0, int(c), 2) for i, c in enumerate(ctx)]
    n_slots = sum(r.max_tokens for r in trace) + 64
    recs, worst = _check(model, trace, [trace[0], trace[1]], max_bs=64, n_slots=n_slots, max_rows=sum(ctx) + 64)
    # iteration 1: every request decodes one row against its long context
    assert recs[1].n_new == [1] * 64 and recs[1].n_ctx == ctx


def test_13b_width_few_hundred_decode_rows(cuda, model):
    """200 requests with short prompts decode together: a 200-row iteration,
    where the QKV Linear takes whole CTA-pair tiles, Attn-Out the single-CTA
    kernel, FC1 pair tiles in stream ranges along K and FC2 (K = 20480)
    three equal k-ranges per pair tile, each with its engine epilogue (K/V
    scatter, GeLU, residual and the folded LayerNorm statistics)."""
    rng = np.random.default_rng(34)
    ctx = [17, 29] + rng.integers(8, 65, 198).tolist()
    trace = [_req(rng, i, 0, int(c), 2) for i, c in enumerate(ctx)]
    n_slots = sum(r.max_tokens for r in trace) + 64
    recs, worst = _check(model, trace, [trace[0], trace[1]], max_bs=256, n_slots=n_slots, max_rows=sum(ctx) + 64)
    assert recs[1].n_new == [1] * 200 and recs[1].n_ctx == ctx


def test_13b_width_decodes_beside_a_prompt(cuda, model):
    """250 decode rows and a 600-token prompt in one iteration (850 rows):
    the FC2 Linear (K = 20480) takes CTA-pair tiles in stream ranges along K
    (the residual with the folded LayerNorm statistics on summed pieces),
    the other Linears whole pair tiles."""
    rng = np.random.default_rng(35)
    ctx = [21, 33] + rng.integers(8, 49, 248).tolist()
    trace = [_req(rng, i, 0, int(c), 2) for i, c in enumerate(ctx)]
    trace.append(_req(rng, 250, 1, 600, 2))
    n_slots = sum(r.max_tokens for r in trace) + 64
    recs, worst = _check(model, trace, [trace[0], trace[1], trace[250]], max_bs=256, n_slots=n_slots,
                         max_rows=sum(ctx) + 64)
    assert sorted(recs[1].n_new) == [1] * 250 + [600]
