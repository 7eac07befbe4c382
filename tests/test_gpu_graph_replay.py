"""The benchmark's own timed configuration against the oracle.

bench.py times steps of write(757) -> reset_positions(42 x 757) ->
attend(757 queries) on rings of 24 heads x 128 and 5,788 slots, one CUDA
graph per set of new tokens (the steps cycle through the sets), the kernels
chained by programmatic dependent launch and the output in bf16.  Here the
same graphs are built by bench.py's own functions and replayed in turn;
after every replay each ring's state, K/V codes and scales must equal the
oracle's bit for bit, and the attention output of three heads (all 757
rows) must be within the attention tolerance plus half a bf16 ulp of the
fp64 oracle over its own cache.  Device-side ring state is what
lets one captured graph be replayed (Runway Characters paper, §4.1)."""
import numpy as np
import pytest
import torch

import synth
from oracle.ring import OracleRing
from replay import compare_attention, compare_cache

pytestmark = pytest.mark.gpu

HEADS = (0, 11, 23)


def test_bench_graph_replays_match_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    R = 3
    dev = torch.device("cuda")
    SETS = 2
    rings, inputs = bench.make_rings(R, dev, sets=SETS)
    prefill = list(synth.single().ops)[0]
    sh = synth.single().shape
    oracles = []
    for r in range(R):
        o = OracleRing(sh.heads, sh.head_dim, sh.n_slots, sh.axis_dims, sh.rope_base)
        o.write(synth.to_f32(prefill.k), synth.to_f32(prefill.v), prefill.pos)
        oracles.append(o)
    host = [[tuple(t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy() for t in inp[:4])
             for inp in per] for per in inputs]
    graphs = [bench.capture(lambda t=t: [bench.step(rings[r], inputs[r][t]) for r in range(R)]) for t in range(SETS)]
    # capture() ran each graph's steps once outside the capture to warm the path
    for t in range(SETS):
        for r in range(R):
            k, v, q, pos = host[r][t]
            oracles[r].write(k, v, pos)
            oracles[r].reset_positions(bench.RESET_D)
    for rep in range(4):
        t = rep % SETS
        graphs[t].replay()
        torch.cuda.synchronize()
        for r in range(R):
            k, v, q, pos = host[r][t]
            o = oracles[r]
            o.write(k, v, pos)
            o.reset_positions(bench.RESET_D)
            assert rings[r].debug_state() == (o.wp, o.n_valid, 0), f"replay {rep} ring {r} state"
            compare_cache(rings[r], o, f"replay {rep} ring {r}")
            out = inputs[r][t][4].float().cpu().numpy()[:, list(HEADS)]
            ref = o.attend(q, pos, heads=list(HEADS))
            compare_attention(out, ref, f"replay {rep} ring {r}", allowance=np.abs(ref) * 2.0 ** -8)
    for g in rings:
        g.close()
