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


# ---------------------------------------------------------------- the online-softmax rescale
#
# The kernel keeps a running maximum m per query row (in base-2 units, the scores times
# log2(e) / sqrt(D)) and rescales the output accumulator and the running sum by 2^(m - m_new)
# only when a key block's row maximum m_new exceeds m by more than 8; smaller rises leave m as
# the reference, so the block's exponentials reach up to 2^8 before the fp16 rounding of P.
# These inputs make the rises happen (keys that grow along the sequence, wide score
# distributions, one huge score late in the sequence), including in the blocks whose keys are
# partly masked (the causal diagonal block, a ragged last block). Before the GPU runs, each
# case proves on the host, from fp64 scores, that the rule fires: the test then pins the
# rescale branch, not only its inputs. (A masked block is always the last block of its row, so
# a rescale after a masked block cannot occur; the rescale inside one can, and is counted.)

def _rescale_events(Q, K, causal):
    """(rescales, rescales inside a partly masked block, rises of at most 2^8) over all query
    rows, following the kernel's rule on fp64 scores."""
    q = Q.numpy().astype(np.float64)
    k = K.numpy().astype(np.float64)
    B, S, H, D = q.shape
    s = np.einsum("bqhd,bkhd->bhqk", q, k) * (np.log2(np.e) / np.sqrt(D))
    pos = np.arange(S)
    if causal:
        s = np.where(pos[None, None, None, :] <= pos[None, None, :, None], s, -np.inf)
    n_kt = (S + 127) // 128
    bm = np.stack([s[..., j * 128:min(S, (j + 1) * 128)].max(-1) for j in range(n_kt)], -1)
    m = bm[..., 0].copy()
    qblk = pos // 128
    rescales = masked = small = 0
    for j in range(1, n_kt):
        seen = (qblk >= j)[None, None, :] if causal else np.ones((1, 1, S), bool)
        part = (qblk == j)[None, None, :] if causal else np.full((1, 1, S), j == n_kt - 1 and S % 128 != 0)
        rise = (bm[..., j] > m + 8) & seen
        small += int(((bm[..., j] > m) & (bm[..., j] <= m + 8) & seen).sum())
        rescales += int(rise.sum())
        masked += int((rise & part).sum())
        m = np.where(rise, bm[..., j], m)
    return rescales, masked, small


RESCALE = [  # (B, S, H, causal, k_ramp, sigma)
    (1, 1000, 2, False, 1.5, 1.0),
    (1, 1000, 2, True, 1.5, 1.0),
    (2, 777, 1, True, 2.5, 1.0),
    (1, 1000, 2, False, 0.0, 2.0),
    (1, 1000, 2, True, 0.0, 2.0),
    (1, 384, 3, False, 2.5, 1.0),
]


@pytest.mark.parametrize("B,S,H,causal,ramp,sigma", RESCALE,
                         ids=[f"{b}x{s}x{h}{'c' if c else ''}_ramp{r}_sd{sd}" for b, s, h, c, r, sd in RESCALE])
def test_rising_maxima_force_the_rescale(tg, B, S, H, causal, ramp, sigma):
    w = workloads.AttnWorkload(f"r_{B}x{S}x{H}", B, S, H, 128, seed=900 + S + H + int(10 * ramp), causal=causal,
                               dist=workloads.Dist("normal", 0.0, sigma), k_ramp=ramp)
    Q, K, V = w.inputs()
    rescales, masked, small = _rescale_events(Q, K, causal)
    assert rescales >= 50, f"only {rescales} rescales: the inputs do not exercise the branch"
    assert small >= 50, f"only {small} rises below the threshold"
    if S % 128 != 0 or causal:
        assert masked >= 5, f"only {masked} rescales inside a partly masked block"
    (Q, K, V), got = _run(tg, w)
    _check(got, oracle.attention(Q, K, V, causal=causal), w.name)
    _status_ok(tg)


@pytest.mark.parametrize("causal", [False, True], ids=["noncausal", "causal"])
def test_huge_late_score_takes_over_the_row(tg, causal):
    """Head 0: every query has 100 in dimension 0 and key 700 (block 5, followed by a ragged
    block of 9 keys) has 100 there too, so its score is about 10^4 / sqrt(128) = 884 while
    the others stay within a few tens: the rescale factor underflows to 0 and each query
    that sees key 700 returns V[700]. Head 1 is left N(0, 1)."""
    B, S, H, s_dom = 1, 777, 2, 700
    w = workloads.AttnWorkload("dominant", B, S, H, 128, seed=960 + int(causal), causal=causal)
    Q, K, V = w.inputs()
    Q[:, :, 0, 0] = 100.0
    K[:, s_dom, 0, 0] = 100.0
    rescales, masked, _ = _rescale_events(Q, K, causal)
    rows_seeing = S - s_dom if causal else S
    assert rescales >= rows_seeing, f"{rescales} rescales for {rows_seeing} rows that see the huge score"
    if causal:
        assert masked >= S - s_dom  # key 700 sits in the diagonal block of queries 640..767
    got = tg.attention(Q.cuda(), K.cuda(), V.cuda(), causal=causal).cpu().numpy()
    ref = oracle.attention(Q, K, V, causal=causal)
    _check(got, ref, "dominant key")
    first = s_dom if causal else 0
    np.testing.assert_allclose(got[0, first:, 0].astype(np.float64),
                               np.broadcast_to(V.numpy()[0, s_dom, 0].astype(np.float64), (S - first, 128)),
                               rtol=1e-3, atol=1e-3)
    _status_ok(tg)


def test_rescale_at_full_length_sampled_rows(tg):
    """4096 positions, 8 heads, keys ramping slowly (every block rises a little, some by more
    than 2^8): sampled rows of every head, first and last positions included."""
    w = workloads.AttnWorkload("ramp_1x4096x8", 1, 4096, 8, 128, seed=970, causal=True, k_ramp=0.3)
    Q, K, V = w.inputs()
    rescales, masked, small = _rescale_events(Q[:, :, :2], K[:, :, :2], True)
    assert rescales >= 50 and small >= 50
    got = tg.attention(Q.cuda(), K.cuda(), V.cuda(), causal=True).cpu().numpy()
    rng = np.random.default_rng(970)
    pos = np.concatenate([[0, 127, 128, 129, 4095], rng.integers(0, 4096, 11)])
    rows = np.array([s * w.H + h for s in pos for h in range(w.H)])
    ref = oracle.attention(Q, K, V, causal=True, rows=rows)
    _check(got.reshape(-1, w.D)[rows], ref, w.name)
    _status_ok(tg)


# ---------------------------------------------------------------- the split last round
#
# Without the mask, when the grid's last round of query blocks (two per SM) is at most half
# full, each of those blocks runs as two CTAs over the two halves of the key blocks, and the
# second to finish merges the partial outputs, maxima and sums. These shapes make the host
# split a known number of blocks: 8 query blocks per head, heads chosen so the blocks fill
# one round of 2 x SMs and leave 16 (the last 16 in launch order).

def _split_heads(per_head_blocks, left_over):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (2 * sms + left_over) // per_head_blocks


@pytest.mark.parametrize("S", [1000, 1024])
def test_split_last_round_every_element(tg, S):
    H = _split_heads(8, 16)
    w = workloads.AttnWorkload(f"split_1x{S}x{H}", 1, S, H, 128, seed=980 + S, k_ramp=0.5)
    Q, K, V = w.inputs()
    dQ, dK, dV = Q.cuda(), K.cuda(), V.cuda()
    got = tg.attention(dQ, dK, dV).cpu().numpy()
    _check(got, oracle.attention(Q, K, V), w.name)
    again = tg.attention(dQ, dK, dV).cpu().numpy()  # the merge is symmetric: same bits every time
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16))
    _status_ok(tg)
