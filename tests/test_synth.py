"""The seeded input generators (no GPU): they draw what the input recipe
says, reproducibly, and hold none of the method's arithmetic."""
import ast
import os

import numpy as np
import torch

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_same_seed_same_values_and_independent_streams():
    a = synth.trits(5, "t", (64, 256))
    assert np.array_equal(a, synth.trits(5, "t", (64, 256)))
    assert not np.array_equal(a, synth.trits(6, "t", (64, 256)))
    # one tensor's shape never shifts another tensor's values
    p1 = synth.problem(9, 1, 32, 256, tag="q")
    p2 = synth.problem(9, 4, 32, 256, tag="q")
    assert np.array_equal(p1.t, p2.t) and np.array_equal(p1.s, p2.s)
    assert np.array_equal(p1.x[0], p2.x[0])


def test_trit_distributions():
    t = synth.trits(1, "t", (512, 4096), synth.SPARSE40)
    f = [(t == v).mean() for v in (-1, 0, 1)]
    assert abs(f[0] - 0.3) < 0.005 and abs(f[1] - 0.4) < 0.005 and abs(f[2] - 0.3) < 0.005
    u = synth.trits(1, "u", (512, 4096), synth.UNIFORM)
    assert all(abs((u == v).mean() - 1 / 3) < 0.005 for v in (-1, 0, 1))
    b = synth.binary(1, "b", (512, 4096))
    assert set(np.unique(b)) == {-1, 1} and abs((b == 1).mean() - 0.5) < 0.005


def test_scale_and_bias_distributions():
    s = synth.scales(2, "s", (4096, 40))
    assert s.dtype == np.float16 and (s >= np.float16(1e-3)).all()
    v = s.astype(np.float64) - 1e-3
    assert abs(np.sqrt(np.pi / 2) * v.mean() - 0.02) < 0.001      # |N(0, 0.02)|: mean = 0.02 sqrt(2/pi)
    su = synth.scales(2, "su", (4096, 40), synth.SCALE_UNIFORM)
    assert su.min() >= np.float16(0.005) and su.max() <= np.float16(0.05)
    b = synth.biases(2, "b", s)
    r = -b.astype(np.float64) / s.astype(np.float64)
    assert b.dtype == np.float16 and r.min() > 0.99 and r.max() < 2.01 and abs(r.mean() - 1.5) < 0.01


def test_code_words_cover_every_code_evenly():
    w = synth.code_words(3, "c", (256, 320))
    q = (w[..., None] >> (2 * np.arange(16, dtype=np.uint32))) & 3
    f = np.bincount(q.ravel(), minlength=4) / q.size
    assert np.all(np.abs(f - 0.25) < 0.005)


def test_bf16_rounding_is_nearest_even():
    rs = np.random.default_rng(0)
    v = np.concatenate([rs.normal(0, 1, 100000), rs.normal(0, 1e-30, 1000), rs.normal(0, 1e30, 1000),
                        [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, np.inf, -np.inf]]).astype(np.float32)
    got = synth.float_to_bf16_bits(v)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    x = synth.activations(4, "x", (4, 4096))
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert abs(xf.std() - 1.0) < 0.03 and abs(xf.mean()) < 0.03


def test_signs_are_pm1():
    s = synth.signs(5, "sg", 4096)
    assert s.dtype == np.int8 and set(np.unique(s)) == {-1, 1} and abs((s == 1).mean() - 0.5) < 0.03


def test_generators_hold_no_method_arithmetic():
    """The one module both sides share imports nothing of either side."""
    tree = ast.parse(open(os.path.join(ROOT, "synth", "__init__.py")).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            mods.add(node.module.split(".")[0])
    assert not mods & {"oracle", "bit_gemv_gemm_gb300"}, mods
