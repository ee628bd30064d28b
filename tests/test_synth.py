"""The seeded input generator: determinism, value sets, document packing."""
import numpy as np

import synth


def test_thread_count_does_not_change_values():
    lib = synth._load()
    a = np.empty(300001, dtype=np.uint16)
    b = np.empty_like(a)
    lib.synth_normal_bf16(a.ctypes.data, a.size, 7, 4, 1)
    lib.synth_normal_bf16(b.ctypes.data, b.size, 7, 4, 13)
    np.testing.assert_array_equal(a, b)
    lib.synth_dyadic_bf16(a.ctypes.data, a.size, 7, 1, -8, 8, 3, 1)
    lib.synth_dyadic_bf16(b.ctypes.data, b.size, 7, 1, -8, 8, 3, 5)
    np.testing.assert_array_equal(a, b)


def test_slices_regenerate_independently():
    full = synth.dyadic_bf16((1000,), 3, 2, -8, 8, 3)
    assert np.array_equal(full[:10], synth.dyadic_bf16((10,), 3, 2, -8, 8, 3))


def test_dyadic_value_sets():
    q = synth.bf16_to_f32(synth.dyadic_bf16((200000,), 1, 1, -8, 8, 3))
    assert set(np.unique(q * 8).astype(int).tolist()) == set(range(-8, 9))
    w = synth.dyadic_f32((100000,), 1, 3, -1, 1, 4)
    assert set(np.unique(w * 16).astype(int).tolist()) == {-1, 0, 1}
    w1 = synth.signed_nonzero_f32((100000,), 0, 3, 8, 3)
    assert set(np.unique(w1 * 8).astype(int).tolist()) == set(range(-8, 0)) | set(range(1, 9))


def test_normal_moments_and_bf16_grid():
    x = synth.bf16_to_f32(synth.normal_bf16((1 << 20,), 2, 4)).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # every value sits on the bf16 grid (low 16 bits of the fp32 pattern are zero)
    assert np.all((x.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)


def test_segments_cover_rows():
    seg = synth.segments(4, 4096, 3, 4)
    for row in seg:
        assert row[0] == 0 and row[-1] == 2
        assert np.all(np.diff(row) >= 0) and set(row.tolist()) == {0, 1, 2}
    seg489 = synth.segments(1, 489, 3, 4)
    assert set(seg489[0].tolist()) == {0, 1, 2}
