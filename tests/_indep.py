"""Test-only independent restatements used to pin the oracle.

These are deliberately written differently from the oracle's C loops: numpy
fancy-index gathers and full-matrix softmax, mpmath at 50 digits, and
torch's fp64 scaled_dot_product_attention.  They serve as brute force /
library cross-checks on small inputs; nothing here is used by the product.
"""
import numpy as np

from paged_kv_cache_218_gb300.workload import bf16_bits_to_f32


def to_f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def gather(cache_bits, table_row, kvh, n, bs=16):
    """Rows 0..n-1 of one sequence for one kv head, via numpy fancy indexing."""
    pos = np.arange(n)
    blocks = np.asarray(table_row)[pos // bs]
    return to_f64(cache_bits[blocks, pos % bs, kvh, :])


def softmax_attention_np(qv, K, V, scale):
    """softmax(scale * K q) V for one query, as a full-matrix numpy expression."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), -np.inf
    x = scale * (K @ qv)
    m = x.max()
    w = np.exp(x - m)
    return (w[:, None] * V).sum(axis=0) / w.sum(), m + np.log(w.sum())


def decode_np(q_bits, kc, vc, bt, lens, scale):
    S, Hq, D = q_bits.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    out = np.zeros((S, Hq, D))
    lse = np.zeros((S, Hq))
    for s in range(S):
        for h in range(Hq):
            K = gather(kc, bt[s], h // G, int(lens[s]))
            V = gather(vc, bt[s], h // G, int(lens[s]))
            out[s, h], lse[s, h] = softmax_attention_np(to_f64(q_bits[s, h]), K, V, scale)
    return out, lse


def attention_mpmath(qv, K, V, scale, dps=50):
    """Attention of one query at ``dps`` decimal digits (mpmath)."""
    import mpmath
    with mpmath.workdps(dps):
        x = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b))
                                             for a, b in zip(qv, k)) for k in K]
        m = max(x)
        w = [mpmath.exp(xi - m) for xi in x]
        tot = mpmath.fsum(w)
        out = [mpmath.fsum(wi * mpmath.mpf(float(v[c])) for wi, v in zip(w, V)) / tot
               for c in range(len(V[0]))]
        lse = m + mpmath.log(tot)
        return np.array([float(o) for o in out]), float(lse)
