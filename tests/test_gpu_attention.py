"""GPU parity of the attention forward (tg_attention_fwd), through the C ABI,
against the fp64 CPU oracle on the same seeded (batch, sequence, head, dim)
inputs: every element of the small workloads and of ragged lengths, sampled
query rows (all heads, first and last positions) of the 4096-token ones and of
shapes whose heads are scheduled in several groups.
Tolerance per element: |gpu - ref| <= 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

RTOL = 1e-2
ATOL = 1e-2


@pytest.fixture(scope="module")
def tg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import tiled_tensor_core_tcgen05_gb300 as m
    torch.cuda.set_device(0)
    return m


def _status_ok(tg):
    st, where = tg.tg_device_status(None)
    assert st == tg.OK, f"device watchdog reported status {st} at wait site {where}"


def _check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = tuple(np.argwhere(bad)[0])
        pytest.fail(f"{what}: {int(bad.sum())}/{bad.size} out of tolerance; first {idx}: gpu={got[idx]} "
                    f"ref={ref[idx]} (max err {err.max():.4g})")


def _run(tg, w):
    Q, K, V = w.inputs()
    O = tg.attention(Q.cuda(), K.cuda(), V.cuda(), causal=w.causal)
    return (Q, K, V), O.cpu().numpy()


@pytest.mark.parametrize("w", [workloads.ATTN_SMALL, workloads.ATTN_SMALL_CAUSAL, workloads.ATTN_RAGGED],
                         ids=lambda w: w.name)
def test_small_workloads_every_element(tg, w):
    (Q, K, V), got = _run(tg, w)
    _check(got, oracle.attention(Q, K, V, causal=w.causal), w.name)
    _status_ok(tg)


SHAPES = [(1, 1, 1, False), (1, 1, 1, True), (1, 127, 2, True), (1, 129, 2, False), (3, 200, 2, True),
          (2, 384, 4, False), (1, 640, 1, True), (1, 257, 3, False)]


@pytest.mark.parametrize("B,S,H,causal", SHAPES, ids=[f"{b}x{s}x{h}{'c' if c else ''}" for b, s, h, c in SHAPES])
def test_shapes_every_element(tg, B, S, H, causal):
    w = workloads.AttnWorkload(f"t_{B}x{S}x{H}", B, S, H, 128, seed=B * 1000 + S + H, causal=causal)
    (Q, K, V), got = _run(tg, w)
    _check(got, oracle.attention(Q, K, V, causal=causal), w.name)
    _status_ok(tg)


@pytest.mark.parametrize("w", [workloads.ATTN_4096, workloads.ATTN_4096_CAUSAL], ids=lambda w: w.name)
def test_full_size_sampled_rows(tg, w):
    (Q, K, V), got = _run(tg, w)
    rng = np.random.default_rng(w.seed)
    pos = np.concatenate([[0, 1, 127, 128, w.S - 1], rng.integers(0, w.S, 27)])
    rows = np.array([(b * w.S + s) * w.H + h for b in range(w.B) for s in pos for h in range(w.H)])
    ref = oracle.attention(Q, K, V, causal=w.causal, rows=rows)
    _check(got.reshape(-1, w.D)[rows], ref, w.name)
    _status_ok(tg)


# (batch, head) pairs whose keys and values exceed 64 MB run as several groups of heads
# (the last one smaller), and a 16384-position sequence: sampled rows of every head, first and
# last positions included
GROUPED = [(1, 8192, 20, True), (3, 4096, 12, False), (1, 16384, 2, True)]


@pytest.mark.parametrize("B,S,H,causal", GROUPED, ids=[f"{b}x{s}x{h}{'c' if c else ''}" for b, s, h, c in GROUPED])
def test_head_groups_sampled_rows(tg, B, S, H, causal):
    w = workloads.AttnWorkload(f"g_{B}x{S}x{H}", B, S, H, 128, seed=7 * B + H, causal=causal)
    (Q, K, V), got = _run(tg, w)
    rng = np.random.default_rng(w.seed)
    pos = np.concatenate([[0, 127, 128, S - 1], rng.integers(0, S, 6)])
    rows = np.array([(b * S + s) * H + h for b in range(B) for s in pos for h in range(H)])
    ref = oracle.attention(Q, K, V, causal=causal, rows=rows)
    _check(got.reshape(-1, w.D)[rows], ref, w.name)
    _status_ok(tg)


def test_causal_first_row_is_the_first_value_exactly(tg):
    w = workloads.ATTN_RAGGED
    (Q, K, V), got = _run(tg, w)
    np.testing.assert_array_equal(got[:, 0].view(np.uint16), V.numpy()[:, 0].view(np.uint16))


def test_repeatable(tg):
    w = workloads.ATTN_SMALL_CAUSAL
    Q, K, V = [t.cuda() for t in w.inputs()]
    a = tg.attention(Q, K, V, causal=True).cpu()
    b = tg.attention(Q, K, V, causal=True).cpu()
    assert torch.equal(a, b)
    _status_ok(tg)
