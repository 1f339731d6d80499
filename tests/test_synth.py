"""The seeded input generators: known-answer vectors and distribution shape (no GPU)."""
import numpy as np

import ftsynth


def test_philox_known_answers():
    # Random123 known-answer vectors for Philox4x32-10
    assert ftsynth.philox4x32_10([0, 0, 0, 0], [0, 0]).tolist() == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert ftsynth.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2).tolist() == [
        0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert ftsynth.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]).tolist() == [
        0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_streams_are_addressable():
    a = ftsynth.normal_bf16(0, 1, 3, 7, 1000)
    b = ftsynth.normal_bf16(0, 1, 3, 7, 600, offset=400)
    assert np.array_equal(a[400:], b)
    assert not np.array_equal(a, ftsynth.normal_bf16(0, 1, 3, 8, 1000))


def test_pool_expert_regenerates_alone():
    L, E, d, f = 2, 3, 64, 32
    for dtype in (0, 1):
        pool = ftsynth.make_pool(0, L, E, d, f, dtype, threads=3)
        bx = ftsynth.expert_bytes(d, f, dtype)
        one = np.empty(bx, dtype=np.uint8)
        ftsynth.fill_pool(one, 0, 1, 1, d, f, dtype, first_layer=1)
        # layer 1 expert 0 of the pool equals a single-expert draw of (layer 1, expert 0)
        assert np.array_equal(pool[(1 * E + 0) * bx:(1 * E + 1) * bx], one)


def test_normal_moments():
    z = ftsynth.normal_f64(0, 1, 0, 0, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01 and abs((z ** 4).mean() - 3) < 0.05
    w = ftsynth.bf16_to_f32(ftsynth.normal_bf16(0, 1, 0, 0, 200000, 0.02))
    assert abs(w.std() - 0.02) < 0.0005


def test_mxfp4_codes_and_scales_distribution():
    d, f = 256, 128
    pool = ftsynth.make_pool(0, 1, 4, d, f, 1, threads=2)
    df = d * f
    bx = ftsynth.expert_bytes(d, f, 1)
    ex = pool[:bx]
    codes = ex[:3 * df // 2]
    nib = np.concatenate([codes & 15, codes >> 4])
    hist = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(hist - 1 / 16) < 0.005)
    scales = ex[3 * df // 2:]
    assert set(np.unique(scales).tolist()) == {119, 120, 121}


def test_ar1_stationary_scale_and_correlation():
    h = ftsynth.bf16_to_f32(ftsynth.ar1_hidden(0, 0, 0, 3000, 64, 0.9)).astype(np.float64)
    tail = h[200:]
    assert abs(tail.std() - 1 / np.sqrt(1 - 0.81)) < 0.1
    c = np.mean(tail[1:] * tail[:-1]) / np.mean(tail * tail)
    assert abs(c - 0.9) < 0.02


def test_bf16_round_trip():
    x = np.array([1.0, -2.5, 3.1415926, 1e-3, 65504.0], dtype=np.float32)
    b = ftsynth.f32_to_bf16(x)
    assert np.array_equal(ftsynth.f32_to_bf16(ftsynth.bf16_to_f32(b)), b)
    assert np.all(np.abs(ftsynth.bf16_to_f32(b) - x) <= np.abs(x) * 2 ** -8)


def test_zipf_routes_distinct_and_skewed():
    r = ftsynth.zipf_routes(0, 0, 128, 64, 8, 1.2, 0, 20, threads=2)
    assert r.shape == (20, 64, 8)
    for row in r.reshape(-1, 8):
        assert len(set(row.tolist())) == 8
    ranks = ftsynth.zipf_ranks(0, 0, 128)
    assert sorted(ranks.tolist()) == list(range(1, 129))
    counts = np.bincount(r.ravel(), minlength=128)
    top = np.argsort(ranks)[:8]
    assert counts[top].sum() > counts.sum() * 0.2  # the 8 best-ranked experts dominate
