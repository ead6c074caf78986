"""The seeded generator: host (numpy) and device-capable (torch) draws agree bit for bit."""
import numpy as np
import torch

import gen


def test_lowbias32_known_values():
    # the hash maps 0 to 0 (all its steps fix zero) and is a bijection on a sample
    assert gen.lowbias32_np(np.array([0], np.uint32))[0] == 0
    x = np.arange(1 << 16, dtype=np.uint32)
    assert np.unique(gen.lowbias32_np(x)).size == x.size


def test_numpy_and_torch_draws_identical():
    for (seed, tag, sub, start, n) in [(0, 4, 5, 0, 1000), (7, 6, (3 << 20) | 17, 123456, 5000),
                                       (2**31 + 5, 1, 2**40 + 9, 2**32 - 100, 200)]:
        a = gen.draws_np(seed, tag, sub, start, n).astype(np.int64)
        b = gen.draws_torch(seed, tag, sub, start, n, "cpu").numpy()
        assert np.array_equal(a, b)


def test_expert_codes_numpy_torch_identical_all_bit_widths():
    for bits in (4, 8, 2):
        s = gen.spec("tiny", weight_bits=bits)
        for which in ("gate", "up", "down"):
            a = gen.expert_codes(s, 5, 1, 3, which)
            b = gen.expert_codes_torch(s, 5, 1, 3, which, "cpu").numpy()
            assert np.array_equal(a, b)
            lo, hi = {4: (-8, 7), 8: (-127, 127), 2: (-2, 1)}[bits]
            assert a.min() == lo and a.max() == hi


def test_hidden_state_rows_independent_and_bf16_exact():
    s = gen.spec("dsv3")
    x, bits = gen.hidden_states(s, 0, 0, 6)
    d = np.zeros(6, np.int64)
    d[3] = 2
    x2, _ = gen.hidden_states(s, 0, 0, 6, d)
    assert np.array_equal(np.delete(x, 3, 0), np.delete(x2, 3, 0))
    assert not np.array_equal(x[3], x2[3])
    xr, _ = gen.hidden_states(s, 0, 0, 6, d, rows=[3, 1])
    assert np.array_equal(xr[0], x2[3]) and np.array_equal(xr[1], x2[1])
    # bf16 values survive a torch bf16 round trip exactly
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(t, x)
    assert abs(float(x.std()) - 1.0) < 0.05
