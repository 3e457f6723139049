"""The seeded input generator: deterministic, sliceable, right distributions."""
import numpy as np
import torch

import moe_synth as S


def test_bf16_rounding_matches_torch():
    v = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 3
    v[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0]     # exact ties and edge values
    ours = S.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(S.bf16_bits_to_f32(ours),
                                  torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_x_slices_match_whole():
    w = S.WORKLOADS["tiny-f32"].scaled(T=600, d=32)
    full = S.x_all(w)
    np.testing.assert_array_equal(S.x_rows(w, 250, 530), full[250:530])
    np.testing.assert_array_equal(S.x_rows(w, 599, 600), full[599:600])
    assert np.array_equal(S.x_all(w), full)          # deterministic


def test_distributions():
    w = S.WORKLOADS["decode-t32-n64-k8"].scaled(d=256, F=128, N=4)
    x = S.to_f64(S.x_all(w), w.dtype)
    assert abs(x.std() - 1.0) < 0.05 and abs(x.mean()) < 0.05
    wg, wu, wd = S.expert_weights(w, 1)
    for a in (wg, wu, wd):
        s = S.to_f64(a, "bf16").std()
        assert abs(s - 0.02) < 0.001
    assert S.gate_weight(w).dtype == np.float32
    assert not np.array_equal(S.expert_weights(w, 0)[0], wg)      # experts differ


def test_zipf_bias_ranks():
    w = S.WORKLOADS["zipf-skew-n128-k8"]
    b = S.gate_bias(w)
    assert b.shape == (128,) and b.dtype == np.float32
    p = np.exp(b.astype(np.float64))
    np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-5)
    ps = np.sort(p)[::-1]
    np.testing.assert_allclose(ps[0] / ps[1], 2 ** 1.2, rtol=1e-4)
    assert S.gate_bias(S.WORKLOADS["tiny-f32"]) is None
