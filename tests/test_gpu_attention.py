"""Ragged attention kernel (orca_attention, through the C ABI) against the
oracle's per-request attention on random K/V slots."""
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


def _run(cuda, dtype, nh, d, batch, seed, gap=3, kv_std=1.0, q_std=1.0):
    """batch: [(L_i, c_i)].  Requests' slots are laid out with `gap` unused
    slots between them (random values there must never be read)."""
    from iteration_level_selective_gb300 import _orca as C
    H = nh * d
    row_off = [0]
    slot_base = []
    s = 5
    for L, c in batch:
        row_off.append(row_off[-1] + L)
        slot_base.append(s)
        s += c + L + gap
    n_slots = s + 7
    N = row_off[-1]
    rng = np.random.default_rng(seed)
    tdt = torch.bfloat16 if dtype == synth.DTYPE_BF16 else torch.float32
    K = torch.from_numpy((rng.standard_normal((nh, n_slots, d)) * kv_std).astype(np.float32)).to(tdt)
    V = torch.from_numpy(rng.standard_normal((nh, n_slots, d)).astype(np.float32)).to(tdt)
    Q = torch.from_numpy((rng.standard_normal((N, H)) * q_std).astype(np.float32)).to(tdt)
    ws_bytes = C.orca_attention_workspace_bytes(len(batch), N, nh, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda)
    out = torch.full((N, H), float("nan"), dtype=tdt, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    Kd, Vd, Qd = K.to(cuda), V.to(cuda), Q.to(cuda)
    C.orca_attention(dtype, nh, d, n_slots, Qd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), out.data_ptr(), row_off,
                     [c for _, c in batch], slot_base, ws.data_ptr(), ws_bytes, status.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.double().cpu().numpy(), Q.double().numpy(), K.double().numpy(), V.double().numpy(), row_off, \
        slot_base


def _check_all(cuda, dtype, nh, d, batch, seed, tol, **kw):
    got, Q, K, V, row_off, slot_base = _run(cuda, dtype, nh, d, batch, seed, **kw)
    worst = 0.0
    for i, (L, c) in enumerate(batch):
        for j in range(L):
            r = row_off[i] + j
            pos = c + j
            sl = slice(slot_base[i], slot_base[i] + pos + 1)
            Kr = K[:, sl, :].transpose(1, 0, 2).reshape(pos + 1, nh * d)   # [T, H], heads concatenated
            Vr = V[:, sl, :].transpose(1, 0, 2).reshape(pos + 1, nh * d)
            want = omodel.attend(Q[r], Kr, Vr, nh)
            worst = max(worst, np.abs(got[r] - want).max() / np.abs(want).max())
    assert worst < tol, worst
    return worst


def test_figure5_batch_fp32(cuda):
    # x1 decode (3 cached), x2 decode (1 cached), x3 prefill 2, x4 prefill 3
    _check_all(cuda, synth.DTYPE_F32, 4, 16, [(1, 3), (1, 1), (2, 0), (3, 0)], seed=1, tol=1e-5, q_std=3.0)


def test_exercise4_batch_fp32_d64(cuda):
    _check_all(cuda, synth.DTYPE_F32, 3, 64, [(37, 0), (9, 0), (1, 120), (1, 15), (1, 64)], seed=2, tol=1e-5,
               q_std=2.0)


@pytest.mark.parametrize("d", [32, 128])
def test_fp32_other_head_dims(cuda, d):
    _check_all(cuda, synth.DTYPE_F32, 2, d, [(20, 0), (1, 700), (5, 3)], seed=3, tol=1e-5)


def test_bf16_d128_chunked_prefill_and_many_splits(cuda):
    # a prefill chunk with cached context, 1- and 2-tile prefills, decodes
    # with 1 .. 12 key splits (split = 256 keys)
    batch = [(100, 50), (17, 0), (1, 0), (1, 255), (1, 256), (1, 1000), (1, 3000), (2, 0)]
    _check_all(cuda, synth.DTYPE_BF16, 4, 128, batch, seed=4, tol=1e-2, q_std=0.3)


def test_bf16_gpt2_heads(cuda):
    batch = [(300, 0), (1, 511), (1, 40), (33, 0), (1, 767)]
    _check_all(cuda, synth.DTYPE_BF16, 12, 64, batch, seed=5, tol=1e-2, q_std=0.3)


def test_decode_stress_full_size_sampled(cuda):
    """13B-shaped heads (40 x 128), 256 decoding requests with cached contexts
    U{1024..4096}, one new token each (one layer of K/V, ~13 GB); 12 sampled
    (request, head) pairs against the oracle."""
    from iteration_level_selective_gb300 import _orca as C
    rng = np.random.default_rng(6)
    nh, d = 40, 128
    ctx = rng.integers(1024, 4097, 256)
    row_off = list(range(257))
    slot_base = np.concatenate([[0], np.cumsum(ctx + 1)[:-1]]).tolist()
    n_slots = int(np.sum(ctx + 1))
    g = torch.Generator(device=cuda)
    g.manual_seed(6)
    K = torch.randn((nh, n_slots, d), device=cuda, generator=g, dtype=torch.bfloat16)
    V = torch.randn((nh, n_slots, d), device=cuda, generator=g, dtype=torch.bfloat16)
    Q = (torch.randn((256, nh * d), device=cuda, generator=g) * 0.2).to(torch.bfloat16)
    ws_bytes = C.orca_attention_workspace_bytes(256, 256, nh, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=cuda)
    out = torch.empty((256, nh * d), dtype=torch.bfloat16, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    C.orca_attention(synth.DTYPE_BF16, nh, d, n_slots, Q.data_ptr(), K.data_ptr(), V.data_ptr(), out.data_ptr(),
                     row_off, ctx.tolist(), slot_base, ws.data_ptr(), ws_bytes, status.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for _ in range(12):
        i, h = int(rng.integers(0, 256)), int(rng.integers(0, nh))
        sl = slice(slot_base[i], slot_base[i] + int(ctx[i]) + 1)
        Kh = K[h, sl].double().cpu().numpy()
        Vh = V[h, sl].double().cpu().numpy()
        qh = Q[i, h * d:(h + 1) * d].double().cpu().numpy()
        want = omodel.attend(qh, Kh, Vh, 1)
        got = out[i, h * d:(h + 1) * d].double().cpu().numpy()
        assert np.abs(got - want).max() / np.abs(want).max() < 1e-2
    del K, V
