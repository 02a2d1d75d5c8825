"""The seeded planted-structure generator (host side)."""

import numpy as np

import synth
from synth import planted as P


def test_splitmix64_known_values():
    # splitmix64 stream from state 0: first outputs of the published generator
    x = np.array([0, 0x9E3779B97F4A7C15], dtype=np.uint64)
    out = P.splitmix64(x)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_normals_moments_and_determinism():
    x = P.normal_bits(3, "k", 1000, 1 << 20)
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.std()) - 1.0) < 5e-3
    assert np.array_equal(x[10:20], P.normal_bits(3, "k", 1010, 10))
    assert not np.array_equal(x[:10], P.normal_bits(4, "k", 1000, 10))
    # values are integers times 2^-16
    assert np.all(np.round(x * 65536) == x * 65536)


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 1.0 + 2**-8 + 2**-20],
                 dtype=np.float32)
    bits = P.f32_to_bf16_bits(f)
    # 1+2^-8 is a tie -> even (1.0); 1+3*2^-8 tie -> 1+2^-6 (even); above tie rounds up
    assert bits.tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC020, 0x3F81]
    assert np.array_equal(P.bf16_bits_to_f32(bits[:1]), np.array([1.0], dtype=np.float32))


def test_row_slices_match_whole_tensor():
    w = synth.WORKLOADS["prefill_1k_d64"].with_(B=2, Hq=4, Hkv=2, Sq=200, Skv=300, window=64)
    t, q, k, v = synth.gen_all(w)
    assert np.array_equal(P.gen_q_rows(w, t, 1, 3, 17, 90), q[1, 3, 17:90])
    assert np.array_equal(P.gen_k_rows(w, t, 1, 1, 33, 250), k[1, 1, 33:250])
    assert np.array_equal(P.gen_v_rows(w, 0, 1, 5, 6), v[0, 1, 5:6])


def test_random_block_count():
    w = synth.WORKLOADS["decode_128k_gqa8"].with_(B=2)
    t = synth.make_tables(w)
    nrb = w.Skv // 64
    assert t.rblk.shape == (2, 8, nrb)
    assert np.all(t.rblk.sum(axis=2) == int(np.floor(0.03 * nrb + 0.5)))


def test_decode_planted_logit_bumps():
    w = synth.WORKLOADS["decode_32k_gqa8"].with_(B=1, Hq=8, Hkv=1, Skv=8192, window=1024)
    t, q, k, v = synth.gen_all(w)
    qf, kf = synth.bf16_bits_to_f64(q)[0], synth.bf16_bits_to_f64(k)[0, 0]
    s = qf @ kf.T / np.sqrt(w.D)
    planted = P.key_planted(w, t, 0, 0, 0, w.Skv)
    assert planted[:64].all() and planted[-1024:].all()
    assert abs(s[:, planted].mean() - 8.0) < 0.5
    assert abs(s[:, ~planted].mean()) < 0.5
    assert 0.8 < s[:, ~planted].std() < 2.0


def test_prefill_window_bump():
    w = synth.WORKLOADS["prefill_1k_d64"]
    t, q, k, v = synth.gen_all(w)
    qf, kf = synth.bf16_bits_to_f64(q)[0, 0], synth.bf16_bits_to_f64(k)[0, 0]
    s = qf @ kf.T / np.sqrt(w.D)
    i = np.arange(300, 1024)
    recent = s[i, i - 100]                   # always inside the previous-or-own segment
    far = s[i, (i - 3 * w.window).clip(min=0)]
    planted_far = P.key_planted(w, t, 0, 0, 0, w.Skv)[(i - 3 * w.window).clip(min=0)]
    assert recent.mean() > 6.0
    assert abs(far[~planted_far].mean()) < 1.0


def test_e4m3_round_matches_worked_values_and_torch():
    # worked values of OCP E4M3 (3 mantissa bits, bias 7): ties go to the even mantissa
    # (-7.75 lies halfway between 7.5 and 8 and goes to 8, mantissa 000)
    x = np.array([1.0, 1.0625, 1.1875, 448.0, 500.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10,
                  -7.75, 0.0, 2.0 ** -6 * 1.0625])
    want = np.array([1.0, 1.0, 1.25, 448.0, 448.0, 2.0 ** -9, 0.0, 2.0 ** -8, -8.0, 0.0,
                     2.0 ** -6])
    assert np.array_equal(synth.e4m3_round(x), want)
    # and torch's own cast (float8_e4m3fn) on bf16-representable values
    rng = np.random.default_rng(0)
    v = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(
        (rng.standard_normal(50000) * 8).astype(np.float32)))
    import torch
    t = torch.tensor(v).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(synth.e4m3_round(v), t)
