"""The seeded input generators: shapes, determinism and the NVFP4
quantiser of the Gaussian workload (checked against values worked by hand
and against torch's float8_e4m3fn rounding)."""
import numpy as np
import torch

from block_scaled_nvfp4_group_gb300 import workloads as wl


def test_shapes_and_seeds():
    d = wl.describe("moe_gate_up")
    assert d["seed"] == 1001 and len(d["shapes"]) == 8
    assert all(40 <= m <= 400 and n == 4096 and k == 7168 for m, n, k in d["shapes"])
    d2 = wl.describe("moe_down")
    assert all(40 <= m <= 400 and n == 7168 and k == 2048 for m, n, k in d2["shapes"])
    assert wl.describe("tiny")["shapes"] == [(64, 256, 256), (128, 256, 256)]
    assert wl.describe("square")["shapes"] == [(4096, 4096, 4096)] * 4


def test_deterministic_and_in_range():
    a = wl.make_groups([(33, 40, 512)], seed=5)[0]
    b = wl.make_groups([(33, 40, 512)], seed=5)[0]
    assert np.array_equal(a.A, b.A) and np.array_equal(a.SFB, b.SFB)
    assert a.A.shape == (33, 256) and a.SFA.shape == (33, 32) and a.B.shape == (40, 256)
    e = (a.SFA >> 3).astype(int) - 7
    assert e.min() >= -4 and e.max() <= 0          # 2^e (1 + m/8), e in [-4, 0]
    assert set(np.unique(a.A & 0xF)) == set(range(16))


def test_e2m1_rounding_hand_values():
    q = np.array([0.0, 0.2, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.1, 7.0, -0.75, -6.5, -0.1])
    want = [0, 0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 8 | 2, 8 | 7, 0]
    assert wl._round_to_e2m1_code(q).tolist() == want


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 500, 4000), 10.0 ** rng.uniform(-4, 2.7, 4000),
                        [0.0, 448.0, 460.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11]])
    code, val = wl._round_to_e4m3(v)
    t = torch.from_numpy(np.minimum(v, 448.0)).to(torch.float8_e4m3fn)
    assert np.array_equal(code, t.view(torch.uint8).numpy())
    assert np.array_equal(val, t.to(torch.float64).numpy())


def test_quantized_workload_reconstructs_gaussian():
    g = wl.make_groups([(64, 32, 256)], seed=3, kind="gaussian")[0]
    assert g.SFA.max() < 0x7F and (g.A.shape == (64, 128))
