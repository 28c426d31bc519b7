"""Gumbel noise for temperature > 0 (oracle side; test infrastructure).

"Deploying FlashRec" (serving parameters): temperature 0 is deterministic
top-k; a temperature above 0 turns the selection into Gumbel top-k, where the
noise only orders the candidates and the returned sequence score does not
include it.  The pages give no formula beyond that; the reading used here
(stated with the others in the design notes):

* ordering key of a candidate with score s:  k = fl32(fl32(s * inv_tau) + g),
  inv_tau = fl32(1 / temperature);
* g ~ Gumbel(0, 1), one independent draw per (request r, step t, beam b,
  token v): g = -ln(-ln(u)), u = (bits23 + 1/2) * 2^-23 from word 0 of
  Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
  easy as 1, 2, 3", SC 2011) at counter (v, b, r, t) and key (seed low
  32 bits, seed high 32 bits); bits23 = word0 >> 9 (so that u is exact in
  float32 and never 0 or 1);
* ln is computed in float32 by the method below, the same operations in the
  same order on both sides, so both take identical ordering decisions.

ln(x), x > 0 normal: x = m * 2^e with m in [sqrt(1/2), sqrt(2)); ln(m) from
the series ln(m) = 2 atanh(z) = 2 (z + z^3/3 + z^5/5 + z^7/7 + z^9/9),
z = (m - 1) / (m + 1), |z| <= 0.1716 (Abramowitz and Stegun 4.1.27; the
dropped terms are below 2e-9); ln x = e * ln2 + ln(m).  Every step is one
float32 operation, round to nearest, no fused multiply-add.
"""
import numpy as np

F32 = np.float32
U32 = np.uint32

# Philox4x32 round multipliers and key increments (Salmon et al., SC 2011)
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85


def _mulhilo(a, b):
    p = a.astype(np.uint64) * np.uint64(b)
    return (p >> np.uint64(32)).astype(U32), (p & np.uint64(0xFFFFFFFF)).astype(U32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds; counters are uint32 arrays (broadcast), the
    key two uint32 scalars.  Returns the four output words."""
    c = [np.asarray(x, dtype=U32) for x in (c0, c1, c2, c3)]
    c = np.broadcast_arrays(*c)
    c = [x.copy() for x in c]
    k0, k1 = np.uint64(k0), np.uint64(k1)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & np.uint64(0xFFFFFFFF)
            k1 = (k1 + np.uint64(PHILOX_W1)) & np.uint64(0xFFFFFFFF)
        hi0, lo0 = _mulhilo(c[0], PHILOX_M0)
        hi1, lo1 = _mulhilo(c[2], PHILOX_M1)
        c = [hi1 ^ c[1] ^ U32(k0), lo1, hi0 ^ c[3] ^ U32(k1), lo0]
    return c


_INV = [F32(1.0), F32(1.0 / 3.0), F32(1.0 / 5.0), F32(1.0 / 7.0), F32(1.0 / 9.0)]
_LN2 = F32(0.6931471805599453)
_SQRT2 = F32(1.4142135623730951)


def ln_f32(x):
    """ln of positive normal float32 values by the atanh series (see module
    notes); float32 array in, float32 array out."""
    x = np.asarray(x, dtype=F32)
    bits = x.view(U32).astype(np.int64)
    e = ((bits >> 23) & 0xFF) - 127
    m = ((bits & 0x7FFFFF) | (127 << 23)).astype(U32).view(F32)      # [1, 2)
    big = m > _SQRT2
    m = np.where(big, (m * F32(0.5)).astype(F32), m).astype(F32)      # exact halving
    e = e + big
    z = ((m - F32(1)).astype(F32) / (m + F32(1)).astype(F32)).astype(F32)
    z2 = (z * z).astype(F32)
    p = _INV[4]
    for c in (_INV[3], _INV[2], _INV[1], _INV[0]):
        p = ((p * z2).astype(F32) + c).astype(F32)
    lnm = ((F32(2) * z).astype(F32) * p).astype(F32)
    return ((e.astype(F32) * _LN2).astype(F32) + lnm).astype(F32)


def gumbel(seed, r, t, b, v):
    """Gumbel(0, 1) draws (float32) for token ids v of beam b, request r,
    step t under the 64-bit seed."""
    seed = int(seed)
    w0 = philox4x32_10(np.asarray(v, dtype=np.int64).astype(U32), U32(b), U32(r), U32(t),
                       seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)[0]
    u = ((w0 >> U32(9)).astype(F32) + F32(0.5)) * F32(2.0 ** -23)    # exact
    y = (-ln_f32(u.astype(F32))).astype(F32)
    return (-ln_f32(y)).astype(F32)


def ordering_keys(s_f32, g_f32, inv_tau_f32):
    """fl32(fl32(s * inv_tau) + g)."""
    return ((np.asarray(s_f32, dtype=F32) * F32(inv_tau_f32)).astype(F32) +
            np.asarray(g_f32, dtype=F32)).astype(F32)


def inv_tau(temperature):
    """fl32(1 / temperature), the division done in float64."""
    return F32(1.0 / float(temperature))
