"""Write oracle_regression.json: the CPU oracles' outputs on tiny seeded cases.

The pages print no worked example with values, so the fixture here is a regression record of the
oracles themselves (they are pinned to mathematics by tests/oracle_pins.py and
tests/mla_oracle_pins.py): any later change to an oracle's arithmetic changes these values, and
regenerating the file is then a deliberate, committed step.  This script calls only ``oracle/``
and the seeded input module; run it from the repository root:

    python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kda_inputs as KI  # noqa: E402
import oracle as O  # noqa: E402
import oracle.mla as OM  # noqa: E402


def cases():
    """The fixture's cases: name -> (function of no arguments returning a dict of arrays)."""
    c = KI.prefill_case("golden", [7, 5], 2, 4, 3, 4, "f32", seed=101, s0_std=0.1, gate=True, conv_width=3)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q, k = unit(c.q), unit(c.k)
    rng = np.random.default_rng(102)
    dO = rng.standard_normal(c.v.shape)

    def recurrent():
        o, s = O.recurrent(q, k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate, cu_seqlens=c.cu_seqlens,
                           scale=c.scale)
        return {"o": o, "final_state": s}

    def chunked():
        o, s = O.chunked(q, k, c.v, c.g, c.beta, initial_state=c.S0, cu_seqlens=c.cu_seqlens, scale=c.scale,
                         chunk=4)
        return {"o": o, "final_state": s}

    def mixer():
        o, s, cs = O.mixer(c.q, c.k, c.v, c.g, c.beta, initial_state=c.S0, gate=c.gate, conv_w=c.conv_w,
                           cu_seqlens=c.cu_seqlens, scale=c.scale, use_qk_l2norm=True)
        return {"o": o, "final_state": s, "conv_state": cs}

    def backward():
        return O.recurrent_backward(q, k, c.v, c.g, c.beta, dO, initial_state=c.S0, cu_seqlens=c.cu_seqlens,
                                    scale=c.scale)

    def mla():
        m = KI.mla_decode_case("golden", 3, 2, 8, 6, [0, 3, 5], seed=103, in_dtype="f32", cache_dtype="bf16",
                               rope_dim=4, theta=100.0)
        out, kc, vc, lens = OM.decode_step(m.q, m.k_new, m.v_new, m.k_cache, m.v_cache, m.cache_len, m.scale,
                                           gate=m.gate, rope_dim=m.rope_dim, theta=m.theta, cache_bf16=True)
        return {"out": out, "k_cache": kc, "v_cache": vc, "cache_len": lens}

    return {"recurrent": recurrent, "chunked": chunked, "mixer": mixer, "backward": backward,
            "mla_decode": mla}


def compute():
    return {name: {k: np.asarray(v, dtype=np.float64).tolist() for k, v in fn().items()}
            for name, fn in cases().items()}


if __name__ == "__main__":
    out = os.path.join(HERE, "oracle_regression.json")
    with open(out, "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (calls only oracle/)", "cases": compute()}, f,
                  separators=(",", ":"))
    print(out)
