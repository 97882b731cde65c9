"""The synthetic workloads have the shapes and load structure they are named for.

The skewed-load layer (T=32768, d=2048, E=128, K=8) routes through a stored
per-expert logit bias: its loads must follow a Zipf law (exponent about 1.2 over
the 124 active experts, no load above T since a token picks an expert once),
with exactly the 4 biased-off experts empty, and must reproduce the loads stored
with the bias when it was written."""
import json

import numpy as np

from oracle import moe_oracle as O
from token_dispatch_grouped_gb300 import inputs as I


def test_workload_shapes():
    shapes = {k: (v.T, v.d, v.E, v.K, v.h) for k, v in I.WORKLOADS.items()}
    assert shapes["tiny"] == (256, 128, 8, 2, 256)
    assert shapes["mixtral"] == (4096, 4096, 8, 2, 14336)
    assert shapes["fine"] == (16384, 2048, 64, 6, 1408)
    assert shapes["skew"] == (32768, 2048, 128, 8, 768)
    assert shapes["long"] == (131072, 4096, 16, 4, 2048)


def test_skewed_layer_loads_follow_zipf_with_empty_experts():
    s = I.WORKLOADS["skew"]
    inp = I.make_layer_inputs(s, seed=0, with_bias=True, parts=("x", "Wg"))
    bias = inp["bias"].numpy().astype(np.float64)
    _, _, ids, _ = O.route(inp["x"], inp["Wg"], s.K, bias)
    load = np.bincount(ids.reshape(-1), minlength=s.E)
    assert load.sum() == s.T * s.K
    # the four experts with bias -1e4 receive nothing, every other expert something
    off = np.nonzero(bias < -1e3)[0]
    assert len(off) == 4 and np.all(load[off] == 0) and (load > 0).sum() == s.E - 4
    assert load.max() <= s.T
    # log-log slope of load against rank over the active experts
    act = np.sort(load[load > 0])[::-1].astype(np.float64)
    slope = -np.polyfit(np.log(np.arange(1, len(act) + 1)), np.log(act), 1)[0]
    assert 1.0 <= slope <= 1.3, slope
    # heavy head: the largest expert takes at least a third of all tokens
    assert act[0] >= s.T / 3
    # the stored loads (written with the bias) are reproduced up to near-ties
    with open(I.SKEW_BIAS_FILE) as f:
        stored = np.asarray(json.load(f)["loads"])
    assert np.abs(stored - load).sum() <= 1e-3 * s.T * s.K
