"""Dense softmax attention in fp64.

Runway Characters paper, §4.3 and Appendix G: every attention call reads the
whole cache (all valid slots) with the cached keys as stored, no causal mask.
Scaled dot-product attention over the valid slots j:

    O_i = sum_j softmax_j(q_i . k_j / sqrt(D)) v_j

computed with a library matmul for the two contractions and a plain softmax in
fp64 (the row maximum is subtracted before exp; this changes nothing but the
rounding).
"""
import numpy as np


def attend_f64(q, k, v):
    """q: [Nq, H, D]; k, v: [H, n, D] (fp64 values) -> O [Nq, H, D] fp64.

    n == 0 is not defined (no key to attend to) and raises."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if k.shape[1] == 0:
        raise ValueError("attention over zero slots is undefined")
    d = q.shape[-1]
    qh = np.transpose(q, (1, 0, 2))                    # [H, Nq, D]
    logits = np.matmul(qh, np.transpose(k, (0, 2, 1))) / np.sqrt(np.float64(d))
    logits -= np.max(logits, axis=-1, keepdims=True)
    p = np.exp(logits)
    p /= np.sum(p, axis=-1, keepdims=True)
    o = np.matmul(p, v)                                # [H, Nq, D]
    return np.transpose(o, (1, 0, 2))
