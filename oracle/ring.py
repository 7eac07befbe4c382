"""The ring KV cache and its three calls, as plain definitions.

Runway Characters paper:
* §4.1 "A ring cache with a device-side write position": one allocation per
  cache; each new chunk goes into circular slots; the write position advances
  with every write.  Each cached token keeps the position it was written with.
* §4.2 "RoPE at write, and a delta rotation at reset": RoPE is applied to the
  new tokens' keys once, before the write; at a reset every cached key is
  dequantised, rotated by R(-d) on the temporal frequencies in fp32 and
  re-quantised; values are not touched (Appendix G).
* §4.3 "FP8 at write": K and V are stored as e4m3; queries are quantised per
  call.
* Appendix G: every attention call reads all the cache's slots.

State: codes uint8 [H, S, D] for K and V, fp32 scales [H, S], the write
position ``wp`` and the count of valid slots ``n_valid``.  A write of N tokens
puts token i into slot (wp + i) mod S, then wp <- (wp + N) mod S and
n_valid <- min(n_valid + N, S).  Slots fill in order 0, 1, 2, ... so the valid
slots are always 0 .. n_valid-1; attention is a sum over them and does not
depend on their order.

Global slots (Introduction, "The model"; Appendix G): a cache may hold
``n_global`` = G slots written once per session, ahead of the window ring.
Slots 0 .. G-1 are the globals; the window ring is slots G .. S-1 (W = S - G
of them).  The globals are written by one call of exactly G tokens, before any
window write; a window write of N tokens then puts token i into slot
G + (wp + i) mod W, wp <- (wp + N) mod W and n_valid <- min(n_valid + N, S).
A reset rotates the valid window slots G .. n_valid-1 only: the global
tokens' positions do not depend on the window.  With G = 0 this is the plain
ring above.  A ring of six latent frames (Appendix G) is the window ring with
W = 6 x 757 and writes of 757 tokens: every frame then fills whole,
consecutive slots and the seventh frame replaces the first.

Fused pre-attention (§4.4; Appendix G): ``write``, ``write_global`` and
``attend`` take an optional ``norm = (gamma, eps)`` that RMS-normalises K
(or Q) per head before RoPE (``oracle.norm``); V is not normalised.

Scales (``scale_mode``).  "token" (the default): one scale per (token,
head), recomputed at write and at reset (absmax, see ``quant``).  "static":
the paper's own scheme (§4.3 "FP8 at write"; Appendix G) -- until
``calibrate`` the ring quantises per token and records each head's absolute
maximum of the K (after RoPE) and V values written; ``calibrate(margin)``
sets one K and one V scale per head from those maxima times the margin,
re-quantises the slots written so far with them (from their dequantised
values, fp32), and from then on writes use them, saturating, and a reset
keeps them and clamps (saturates) the rotated keys.  A reset before the
calibration is refused: the paper calibrates on entering the seventh step and
resets every 42.
"""
import numpy as np

from . import norm, quant, rope
from .attention import attend_f64


class OracleRing:
    def __init__(self, heads, head_dim, n_slots, axis_dims, base=10000.0, n_global=0, scale_mode="token"):
        if sum(axis_dims) != head_dim or any(d % 2 for d in axis_dims):
            raise ValueError("axis_dims must be even and sum to head_dim")
        self.H, self.D, self.S = int(heads), int(head_dim), int(n_slots)
        self.G = int(n_global)
        if not 0 <= self.G < self.S:
            raise ValueError("n_global must leave at least one window slot")
        self.W = self.S - self.G
        self.globals_written = False
        if scale_mode not in ("token", "static"):
            raise ValueError("scale_mode is 'token' or 'static'")
        self.scale_mode = scale_mode
        self.static = None                                # (k_scale, k_inv, v_scale, v_inv), [H] each
        self.cal_amax_k = np.zeros(int(heads), np.float32)
        self.cal_amax_v = np.zeros(int(heads), np.float32)
        self.axis_dims = tuple(int(d) for d in axis_dims)
        self.base = float(base)
        self.k_codes = np.zeros((self.H, self.S, self.D), np.uint8)
        self.v_codes = np.zeros((self.H, self.S, self.D), np.uint8)
        self.k_scale = np.zeros((self.H, self.S), np.float32)
        self.v_scale = np.zeros((self.H, self.S), np.float32)
        self.wp = 0
        self.n_valid = 0

    # -- write ---------------------------------------------------------------
    def slots_for(self, n_new):
        return self.G + (self.wp + np.arange(n_new)) % self.W

    def _store(self, k, v, pos, slots, norm_k=None):
        """RMS norm of K (if asked), RoPE on K (fp32), e4m3 of K and V
        (per-token absmax scales, or the fixed per-head ones once
        calibrated), into ``slots``."""
        if norm_k is not None:
            k = norm.rms_norm_bf16(k, norm_k[0], norm_k[1])
        kr = rope.rope_f32(k, pos, self.axis_dims, self.base)
        if self.static is None:
            kc, ks = quant.quantize_rows(kr)
            vc, vs = quant.quantize_rows(v)
            if self.scale_mode == "static":
                self.cal_amax_k = np.maximum(self.cal_amax_k, np.abs(kr).max(axis=(0, 2)))
                self.cal_amax_v = np.maximum(self.cal_amax_v, np.abs(v).max(axis=(0, 2)))
        else:
            k_scale, k_inv, v_scale, v_inv = self.static
            n = kr.shape[0]
            kc = quant.quantize_rows_fixed(kr, np.broadcast_to(k_inv, (n, self.H)))
            vc = quant.quantize_rows_fixed(v, np.broadcast_to(v_inv, (n, self.H)))
            ks = np.broadcast_to(k_scale, (n, self.H))
            vs = np.broadcast_to(v_scale, (n, self.H))
        self.k_codes[:, slots, :] = np.transpose(kc, (1, 0, 2))
        self.v_codes[:, slots, :] = np.transpose(vc, (1, 0, 2))
        self.k_scale[:, slots] = ks.T
        self.v_scale[:, slots] = vs.T

    def write(self, k, v, pos, norm_k=None):
        """k, v: float32 [N, H, D] (bf16 values); pos: int [N, n_axes].
        Window write.  Returns the slot index of each token."""
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        n = k.shape[0]
        if not 1 <= n <= self.W:
            raise ValueError("a write must carry 1 .. n_slots - n_global tokens")
        if self.G and not self.globals_written:
            raise ValueError("the global slots are written before the first window write")
        slots = self.slots_for(n)
        self._store(k, v, pos, slots, norm_k)
        self.wp = int((self.wp + n) % self.W)
        self.n_valid = int(min(self.n_valid + n, self.S))
        return slots

    def write_global(self, k, v, pos, norm_k=None):
        """The G global tokens of the session, once, into slots 0 .. G-1
        (same arithmetic as a window write).  Returns their slots."""
        k = np.asarray(k, np.float32)
        v = np.asarray(v, np.float32)
        if self.G == 0 or k.shape[0] != self.G:
            raise ValueError("a global write carries exactly n_global tokens")
        if self.globals_written or self.n_valid:
            raise ValueError("the global slots are written once, before any window write")
        slots = np.arange(self.G)
        self._store(k, v, pos, slots, norm_k)
        self.globals_written = True
        self.n_valid = self.G
        return slots

    # -- calibration (scale_mode "static") --------------------------------------
    def calibrate(self, margin=1.5):
        """Fix the per-head K and V scales from the recorded maxima times
        ``margin`` and re-quantise the valid slots with them."""
        if self.scale_mode != "static" or self.static is not None:
            raise ValueError("calibrate once, on a ring with scale_mode 'static'")
        if self.n_valid == 0:
            raise ValueError("calibrate after the first write")
        k_scale, k_inv = quant.static_scale(self.cal_amax_k, margin)
        v_scale, v_inv = quant.static_scale(self.cal_amax_v, margin)
        n = self.n_valid
        for codes, scales, sc, iv in ((self.k_codes, self.k_scale, k_scale, k_inv),
                                      (self.v_codes, self.v_scale, v_scale, v_inv)):
            x = quant.dequantize_rows(codes[:, :n], scales[:, :n])
            codes[:, :n] = quant.quantize_rows_fixed(x, np.broadcast_to(iv[:, None], (self.H, n)))
            scales[:, :n] = sc[:, None]
        self.static = (k_scale, k_inv, v_scale, v_inv)

    # -- reset ---------------------------------------------------------------
    def reset_positions(self, d):
        """Rotate every valid window key by R(-d) on the temporal axis
        (axis 0), in fp32, and re-quantise it with a fresh absmax scale.
        Global keys are not touched."""
        if self.scale_mode == "static" and self.static is None:
            raise ValueError("a ring with scale_mode 'static' is calibrated before its first reset")
        lo, hi = self.G, self.n_valid
        if hi <= lo:
            return
        c, s = rope.delta_cos_sin_f32(d, self.axis_dims[0], self.base)
        k = quant.dequantize_rows(self.k_codes[:, lo:hi], self.k_scale[:, lo:hi])
        k = rope.rotate_temporal_f32(k, c, s, self.axis_dims[0])
        if self.static is None:
            codes, scale = quant.quantize_rows(k)
            self.k_scale[:, lo:hi] = scale
        else:
            # the same per-head scale; rotated values beyond the range saturate
            codes = quant.quantize_rows_fixed(k, np.broadcast_to(self.static[1][:, None], (self.H, hi - lo)))
        self.k_codes[:, lo:hi] = codes

    # -- attend --------------------------------------------------------------
    def quantized_queries(self, q, q_pos, norm_q=None):
        """RMS norm (if asked), RoPE (fp32), then per-token-per-head e4m3:
        (codes [Nq,H,D], scale [Nq,H])."""
        q = np.asarray(q, np.float32)
        if norm_q is not None:
            q = norm.rms_norm_bf16(q, norm_q[0], norm_q[1])
        return quant.quantize_rows(rope.rope_f32(q, q_pos, self.axis_dims, self.base))

    def attend(self, q, q_pos, heads=None, rows=None, norm_q=None):
        """fp64 attention of the quantised queries over the valid slots.

        q: float32 [Nq, H, D] (bf16 values); q_pos: int [Nq, n_axes].
        ``heads`` / ``rows`` restrict the output to some heads / query rows
        (for sampled checks); the result is [len(rows), len(heads), D]."""
        qc, qs = self.quantized_queries(q, q_pos, norm_q)
        heads = np.arange(self.H) if heads is None else np.asarray(heads)
        rows = np.arange(qc.shape[0]) if rows is None else np.asarray(rows)
        qh = quant.dequantize_rows_f64(qc[rows][:, heads], qs[rows][:, heads])
        n = self.n_valid
        kh = quant.dequantize_rows_f64(self.k_codes[heads, :n], self.k_scale[heads, :n])
        vh = quant.dequantize_rows_f64(self.v_codes[heads, :n], self.v_scale[heads, :n])
        return attend_f64(qh, kh, vh)
