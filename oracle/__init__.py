"""CPU oracle for the write-time FP8 ring KV cache and the attention that reads it.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, table or constant generator with the CUDA library; the two meet only
through the seeded inputs of ``synth``.

Source: "Runway Characters: Serving a 57B Video Diffusion Transformer for
Real-Time Conversation" (arXiv:2611.05642), Introduction ("The model": global
slots and the window of six latent frames), §4.1 (ring cache with a
device-side write position), §4.2 (RoPE at write, delta rotation at reset),
§4.3 (FP8 at write), Appendix G (cache update and position reset).

Every function is written from the plain definition of what it computes:

* ``e4m3``  -- the OCP E4M3 ("FN") code table and a round-to-nearest-even,
  saturating encoder.
* ``quant`` -- per-token-per-head absmax quantisation to e4m3, and the
  paper's per-head scales fixed once per session (margin x amax, saturating).
* ``rope``  -- RoPE frequencies, the fp32 cos/sin tables, RoPE in fp32 and in
  fp64, the delta rotation R(-d).
* ``ring``  -- the ring of slots with its write position, the optional global
  slots ahead of it (written once, never rotated), the scale mode (per token,
  or per head fixed by ``calibrate``), and the whole call sequence
  (write_global / write / calibrate / reset_positions / attend).
* ``attention`` -- dense softmax attention in fp64.
* ``norm``  -- RMS normalisation of Q and K ahead of RoPE (the fused
  pre-attention step), each step one fixed rounding.

Parity pins (tests/test_oracle_*.py) tie each function to something other than
itself: closed forms, invariants, brute force, the library float8 cast of
PyTorch.  No function here is "parity unpinned".
"""
