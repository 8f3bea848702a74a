"""CPU check of the wide-range weight patterns used by the GPU parity tests."""
import numpy as np

import oracle
import synth
import wide_range as wr


def test_wide_range_patterns_decode_as_intended():
    """The wide-range weight patterns: the oracle decodes code 1 (zero) exactly where
    they put it and +d elsewhere."""
    g = synth.rng(2201)
    N, K = 3, 256
    w = wr.all_code2(g, N, K)
    wr.set_code(w, N, K, 1, 77, 1)
    wr.set_code(w, N, K, 2, 255, 0)
    dq = oracle.dequantize(w, N, K)
    d = np.array([[oracle.block_scale_bits(w.reshape(-1, 18)[r * 4 + b]) for b in range(4)]
                  for r in range(N)])
    dv = oracle.halves_to_double(d)
    want = np.repeat(dv, 64, axis=1)
    want[1, 77] = 0.0
    want[2, 255] = -dv[2, 3]
    assert np.array_equal(dq, want)
