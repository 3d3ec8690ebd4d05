"""orca_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (its scratch is a fixed device array inside the
library).  Checked against orca_attention, whose scratch the caller
allocates, on two calls in a row: both run the same kernels on the same
inputs and the key-split merge goes in split order, so the outputs must be
identical bit for bit; both are also checked against the oracle's
per-request attention.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import numpy as np
import pytest

import synth
from oracle import model as omodel

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda(liborca):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _batch(cuda, seed, nh, d, batch):
    rng = np.random.default_rng(seed)
    row_off, slot_base, s = [0], [], 3
    for L, c in batch:
        row_off.append(row_off[-1] + L)
        slot_base.append(s)
        s += c + L + 2
    n_slots = s
    K = torch.from_numpy(rng.standard_normal((nh, n_slots, d)).astype(np.float32)).to(torch.bfloat16).to(cuda)
    V = torch.from_numpy(rng.standard_normal((nh, n_slots, d)).astype(np.float32)).to(torch.bfloat16).to(cuda)
    Q = torch.from_numpy((rng.standard_normal((row_off[-1], nh * d)) * 0.3).astype(np.float32)).to(
        torch.bfloat16).to(cuda)
    return Q, K, V, row_off, [c for _, c in batch], slot_base, n_slots


def test_noalloc_matches_caller_scratch_entry_two_calls(cuda):
    from iteration_level_selective_gb300 import _orca as C
    nh, d = 8, 128
    st = torch.cuda.current_stream().cuda_stream
    # two different batches; both use key splits (partials and counters in scratch)
    batches = [[(40, 0), (1, 900), (1, 3000), (17, 5), (1, 1)],
               [(1, 2500), (3, 0), (1, 700), (64, 30)]]
    for call, batch in enumerate(batches):
        Q, K, V, row_off, ctx, slot_base, n_slots = _batch(cuda, 100 + call, nh, d, batch)
        N = row_off[-1]
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        ws_bytes = C.orca_attention_workspace_bytes(len(batch), N, nh, d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda)
        ref = torch.empty((N, nh * d), dtype=torch.bfloat16, device=cuda)
        C.orca_attention(synth.DTYPE_BF16, nh, d, n_slots, Q.data_ptr(), K.data_ptr(), V.data_ptr(), ref.data_ptr(),
                         row_off, ctx, slot_base, ws.data_ptr(), ws_bytes, status.data_ptr(), st)
        out = torch.full((N, nh * d), float("nan"), dtype=torch.bfloat16, device=cuda)
        C.orca_attention_noalloc(synth.DTYPE_BF16, nh, d, n_slots, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                 out.data_ptr(), row_off, ctx, slot_base, status.data_ptr(), st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), call
        # and both are the attention the oracle computes, row by row
        o = out.double().cpu().numpy()
        Qh, Kh, Vh = Q.double().cpu().numpy(), K.double().cpu().numpy(), V.double().cpu().numpy()
        worst = 0.0
        for i, (L, c) in enumerate(batch):
            for j in range(L):
                r, pos = row_off[i] + j, c + j
                sl = slice(slot_base[i], slot_base[i] + pos + 1)
                Kr = Kh[:, sl, :].transpose(1, 0, 2).reshape(pos + 1, nh * d)
                Vr = Vh[:, sl, :].transpose(1, 0, 2).reshape(pos + 1, nh * d)
                want = omodel.attend(Qh[r], Kr, Vr, nh)
                worst = max(worst, np.abs(o[r] - want).max() / np.abs(want).max())
        assert worst < 1e-2, (call, worst)


def test_noalloc_rejects_batches_beyond_its_scratch(cuda):
    """A batch whose work records and key-split partials exceed the fixed
    scratch is refused before any launch (real, valid buffers are passed
    all the same)."""
    from iteration_level_selective_gb300 import _orca as C
    nh, d, n = 40, 128, 32          # 32 decode rows of 40 heads x 128: ~11 MiB of partials
    Q, K, V, row_off, ctx, slot_base, n_slots = _batch(cuda, 7, nh, d, [(1, 150)] * n)
    out = torch.empty((n, nh * d), dtype=torch.bfloat16, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    with pytest.raises(C.OrcaError) as ei:
        C.orca_attention_noalloc(synth.DTYPE_BF16, nh, d, n_slots, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                 out.data_ptr(), row_off, ctx, slot_base, status.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert ei.value.code == C.ORCA_EBATCH
