"""The seeded generator: determinism, known SplitMix64 outputs and the value
ranges the workload definition asks for."""
import numpy as np

from synth import generate as S


def test_splitmix64_reference_outputs():
    """First outputs of SplitMix64 seeded with 0 (published test vector of
    Vigna's splitmix64.c): 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4."""
    r = S.raw64(0, 0, 2)
    assert int(r[0]) == 0xE220A8397B1DCDAF
    assert int(r[1]) == 0x6E789E6AA1B965F4


def test_counter_slices_are_independent():
    k = S.stream_key(1, 2, 3)
    full = S.raw64(k, 0, 100)
    assert np.array_equal(full[37:60], S.raw64(k, 37, 23))


def test_expert_value_ranges():
    ex = S.expert(S.SEED, 0, 5, 256, 128, 4)
    codes, sc, bi = ex["gate"]
    assert codes.shape == (128, 128) and sc.shape == (128, 4)
    s = S.bf16_bits_to_f32(sc).astype(np.float64)
    b = S.bf16_bits_to_f32(bi).astype(np.float64)
    assert s.min() >= 0.005 * (1 - 2**-8) and s.max() <= 0.02 * (1 + 2**-8)
    ratio = b / s
    assert ratio.min() >= -8.8 * (1 + 2**-7) and ratio.max() <= -7.2 * (1 - 2**-7)
    nib = np.concatenate([codes & 15, codes >> 4]).ravel()
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.8 * nib.size / 16 and counts.max() < 1.2 * nib.size / 16
    ex2 = S.expert(S.SEED, 0, 5, 256, 128, 2)
    b2 = S.bf16_bits_to_f32(ex2["gate"][2]).astype(np.float64) / S.bf16_bits_to_f32(ex2["gate"][1])
    assert b2.min() >= -1.65 * (1 + 2**-7) and b2.max() <= -1.35 * (1 - 2**-7)


def test_normals_and_router_scale():
    z = S.normal(S.stream_key(9), 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    R = S.bf16_bits_to_f32(S.router(S.SEED, 0, 16, 256))
    assert abs(R.std() - 0.02) < 0.002


def test_reuse_trace_statistics():
    tr = S.reuse_trace(S.SEED, 0, 256, 512, 4)
    for t in range(256):
        assert len(set(tr[t].tolist())) == 4
    same = np.mean(tr[1:] == tr[:-1])
    assert 0.2 < same < 0.34  # p = 0.27 per slot, plus rare fresh re-draws
