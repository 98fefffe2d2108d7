"""Workload definitions and the algorithmic flop/byte counts the benchmark
reports, pinned to the worked traffic example of "TileLang: writing LLM GPU
kernels by thinking in tiles", section 2, "A back-of-the-envelope calculation"."""
import os

import numpy as np
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = int(v)
    return out


def test_traffic_worked_example():
    g = _kv("traffic_4096.txt")
    w = workloads.custom(g["M"], g["N"], g["K"], seed=0)
    assert w.flops() == g["flops"]
    assert round(w.flops() / 1e9) == g["flops_page_billions"]
    assert w.bytes() == g["ideal_bytes"] == 3 * g["matrix_bytes"]
    assert g["matrix_bytes"] // 2 ** 20 == g["matrix_page_mb"]
    assert g["ideal_bytes"] // 2 ** 20 == g["ideal_page_mb"]
    # naive: every output reads a K-row of A and a K-column of B, 2 bytes each
    assert g["M"] * g["N"] * (2 * g["K"]) * 2 == g["naive_input_bytes"]
    assert round(g["naive_input_bytes"] / 1e9) == g["naive_page_gb"]


def test_five_workloads_shapes():
    names = [w.name for w in workloads.ALL]
    assert len(set(names)) == 5
    assert (workloads.SQUARE_8192.M, workloads.SQUARE_8192.N, workloads.SQUARE_8192.K) == (8192,) * 3
    d = workloads.DECODE
    assert (d.M, d.N, d.K) == (16, 28672, 8192)
    assert d.bytes() == 2 * (16 * 8192 + 8192 * 28672 + 16 * 28672) == 470_941_696
    r = workloads.RAGGED_GELU
    assert all(x % 64 for x in (r.M, r.N, r.K)) and r.gelu and r.has_bias


def test_inputs_are_seeded_and_fp16():
    w = workloads.custom(33, 17, 9, seed=5, bias=workloads.Dist("uniform", -0.1, 0.1))
    A1, B1, b1 = w.inputs()
    A2, B2, b2 = w.inputs()
    assert A1.dtype == B1.dtype == b1.dtype == torch.float16
    assert torch.equal(A1, A2) and torch.equal(B1, B2) and torch.equal(b1, b2)
    assert A1.shape == (33, 9) and B1.shape == (9, 17) and b1.shape == (17,)
    assert float(A1.abs().max()) <= 1.0 and float(b1.abs().max()) <= 0.1
    other = workloads.custom(33, 17, 9, seed=6).inputs()[0]
    assert not torch.equal(A1, other)


def test_integer_distribution_is_integer():
    w = workloads.custom(20, 20, 20, seed=1, dist=workloads.Dist("int", -2, 2))
    A, B, _ = w.inputs()
    a = A.float().numpy()
    assert np.array_equal(a, np.round(a)) and a.min() >= -2 and a.max() <= 2


def test_w4_workload_packing_and_bytes():
    w = workloads.W4Workload("t", 3, 16, 256, seed=9)
    A, Bq, s, b = w.inputs()
    assert A.shape == (3, 256) and Bq.shape == (16, 128) and Bq.dtype == torch.uint8
    assert s.shape == (2, 16) and s.dtype == torch.float16 and b is None
    A2, Bq2, s2, _ = w.inputs()
    assert torch.equal(Bq, Bq2) and torch.equal(s, s2)
    d = workloads.DECODE_W4
    assert d.bytes() == 2 * 16 * 8192 + 8192 * 28672 // 2 + 2 * 64 * 28672 + 2 * 16 * 28672


def test_attention_workloads_are_seeded_and_sized():
    w = workloads.ATTN_SMALL
    Q, K, V = w.inputs()
    assert Q.shape == K.shape == V.shape == (1, 256, 2, 128) and Q.dtype == torch.float16
    Q2, K2, V2 = w.inputs()
    assert torch.equal(Q, Q2) and torch.equal(V, V2) and not torch.equal(Q, K)
    big = workloads.ATTN_4096
    assert big.flops() == 4 * 32 * 128 * 4096 * 4096
    assert workloads.ATTN_4096_CAUSAL.flops() == 4 * 32 * 128 * (4096 * 4097 // 2)
    assert big.bytes() == 8 * 4096 * 32 * 128


def test_softmax_workloads():
    w = workloads.SOFTMAX_RAGGED
    (X,) = w.inputs()
    (X2,) = w.inputs()
    assert X.shape == (1000, 1030) and X.dtype == torch.float16 and torch.equal(X, X2)
    assert workloads.SOFTMAX_4096.bytes() == 4 * 32768 * 4096


def test_key_ramp_scales_keys_by_position_and_leaves_q_v_alone():
    plain = workloads.AttnWorkload("p", 1, 300, 2, 128, seed=77)
    ramp = workloads.AttnWorkload("r", 1, 300, 2, 128, seed=77, k_ramp=2.0)
    Qp, Kp, Vp = plain.inputs()
    Qr, Kr, Vr = ramp.inputs()
    assert torch.equal(Qp, Qr) and torch.equal(Vp, Vr)
    scale = 1.0 + 2.0 * torch.arange(300, dtype=torch.float32) / 128.0
    expect = (Kp.to(torch.float32) * scale.view(1, 300, 1, 1)).to(torch.float16)
    assert torch.equal(Kr, expect)


def test_fp4_workload_draws_every_code_and_int4_draws_are_unchanged():
    w = workloads.W4Workload("f", 4, 64, 256, seed=3, fmt="fp4")
    A, Bq, s, bias = w.inputs()
    codes = np.concatenate([(Bq.numpy() & 0xF).ravel(), (Bq.numpy() >> 4).ravel()])
    assert set(codes.tolist()) == set(range(16)) and w.fmt_code == 1
    i = workloads.W4Workload("i", 4, 64, 256, seed=3)
    A2, Bq2, _, _ = i.inputs()
    assert torch.equal(A, A2) and i.fmt_code == 0
    g = torch.Generator().manual_seed(3)
    workloads.Dist("normal", 0.0, 1.0).draw((4, 256), g)
    q = torch.randint(-8, 8, (64, 256), generator=g, dtype=torch.int16)
    u = (q & 0xF).to(torch.uint8)
    assert torch.equal(Bq2, (u[:, 0::2] | (u[:, 1::2] << 4)).contiguous())
