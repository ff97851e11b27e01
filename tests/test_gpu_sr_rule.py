"""Blackwell's stochastic-rounding conversion, exactly as the SR kernels apply
it (nvfp4moe_sr_e4m3x4: cvt.rs with the library's draw convention), held to
the oracle's rule ("Re-quantization with stochastic rounding": round up iff
R < floor(f 2^16), oracle.formats.sr_code) draw by draw:
  * every draw R in [0, 2^16) for values at chosen positions f 2^16 of a gap
    in every E4M3 binade: the subnormal gaps, the first and last gap of each
    normal binade, the top gap below 448, at positions k and k + 1/2 (the
    dropped bits below the top 16 must not matter), negative values included;
  * the draws at and around the threshold floor(f 2^16) for the rest;
  * zeros, signed zeros and saturating values.
The second value of each pair reads the bit-reversed draw; the test builds
each value's draw R from the words it passes, so all four lanes of the
conversion are covered."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.philox import bitrev16
from precision_moe_numerics_nvfp4_gb300 import nvfp4moe as N
from tests.gpu_helpers import check_status, dev, gempty

pytestmark = pytest.mark.gpu

MAGS = F.E4M3_TABLE[0]
KS = [0, 1, 2, 0x00FF, 0x5555, 0x7FFF, 0x8000, 0x8001, 0xAAAA, 0xFFFE, 0xFFFF]


def _gaps():
    """(a, b) pairs of neighbouring E4M3 magnitudes: every subnormal gap, the
    first and last gap of every normal binade, the top gap."""
    pairs = [(MAGS[i], MAGS[i + 1]) for i in range(8)]                      # 0 .. 2^-6, step 2^-9
    for e in range(-6, 9):
        lo, hi = 2.0 ** e, 2.0 ** e * 15 / 8
        i = int(np.searchsorted(MAGS, lo))
        j = int(np.searchsorted(MAGS, hi))
        if i + 1 < len(MAGS):
            pairs.append((MAGS[i], MAGS[i + 1]))
        if j + 1 < len(MAGS):
            pairs.append((MAGS[j], MAGS[j + 1]))
    pairs.append((MAGS[-2], MAGS[-1]))                                        # 416 .. 448
    return sorted(set(pairs))


def _value(a, b, k):
    v = a + (b - a) * k / 65536.0
    assert np.float32(v) == v, (a, b, k)
    return v


def _draws_of(words):
    lo, hi = words & 0xFFFF, words >> 16
    return np.stack([lo, bitrev16(lo), hi, bitrev16(hi)], axis=1).reshape(-1).astype(np.int64)


def _run(x, words):
    xt = gempty(x.size, dtype=torch.float32, device=dev())
    xt.copy_(torch.from_numpy(x.astype(np.float32)))
    wt = gempty(words.size, dtype=torch.int32, device=dev())
    wt.copy_(torch.from_numpy(words.astype(np.uint32).view(np.int32)))
    out = gempty(x.size, dtype=torch.uint8, device=dev())
    N.nvfp4moe_sr_e4m3x4(xt, wt, words.size, out)
    check_status()
    return out.cpu().numpy()


def _check(x, words):
    got = _run(x, words)
    want = F.sr_code(x.astype(np.float32), F.E4M3_TABLE, _draws_of(words))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), int(_draws_of(words)[i]), int(got[i]), int(want[i])) for i in bad[:8]]


def test_every_draw_for_values_in_every_binade():
    gaps = _gaps()
    vals = []
    for n, (a, b) in enumerate(gaps):
        k = KS[(n * 5 + 3) % len(KS)]
        vals.append(_value(a, b, k))
        vals.append(_value(a, b, min(k + 0.5, 65535.5)))   # bits below the top 16 dropped bits
    vals += [-vals[3], -vals[20], -vals[-1]]                 # negative values
    while len(vals) % 4:
        vals.append(vals[len(vals) % 7])
    vals = np.array(vals, dtype=np.float64)
    G = vals.size // 4
    r = np.arange(65536, dtype=np.uint64)
    words = (r | (r << np.uint64(16))).astype(np.uint64)    # every draw in every lane
    x = np.tile(vals.reshape(G, 4), (65536, 1)).reshape(-1)
    w = np.repeat(words, G)
    _check(x, w)


def test_threshold_draws_for_every_gap_position():
    rng = np.random.default_rng(7)
    xs, ds = [], []
    for a, b in _gaps():
        for k in KS:
            for kk in (k, k + 0.5):
                if kk >= 65536:
                    continue
                v = _value(a, b, kk)
                d = int(np.floor(kk))
                for R in sorted({0, 1, max(d - 2, 0), max(d - 1, 0), d, min(d + 1, 65535), 65535}):
                    xs.append(v if rng.random() < 0.8 else -v)
                    ds.append(R)
    # zeros, signed zeros and saturating values
    for v in (0.0, -0.0, 448.0, -448.0, 449.0, 460.0, 1e6, -3e9):
        for R in (0, 1, 32768, 65535):
            xs.append(v)
            ds.append(R)
    while len(xs) % 4:
        xs.append(0.0)
        ds.append(0)
    x = np.array(xs, dtype=np.float64)
    ds = np.array(ds, dtype=np.uint32).reshape(-1, 4)
    # lanes 0 and 2 read U_a, U_b as they are, lanes 1 and 3 bit-reversed: one
    # pass gives lanes 0 / 2 their chosen draws, a second (reversed words)
    # lanes 1 / 3; every lane is checked against the oracle in both
    _check(x, ds[:, 0].astype(np.uint64) | (ds[:, 2].astype(np.uint64) << np.uint64(16)))
    _check(x, bitrev16(ds[:, 1]).astype(np.uint64) | (bitrev16(ds[:, 3]).astype(np.uint64) << np.uint64(16)))
