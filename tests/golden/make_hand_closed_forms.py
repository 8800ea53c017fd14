"""Writes hand_closed_forms.json: hand-derived closed forms, evaluated with math only.

The pages print no worked numeric example, so these fixtures are small cases
whose answers follow by hand from the definitions: the 656-byte row layout
(FlashInfer PR #4802 "Refactor Sparse MLA SM120", review note on the DSv3.2
per-token KV layout) and the sink softmax (vLLM PR #57673, Test Result
section: attn_sink + topk_length).  No oracle or CUDA code is involved.
Run: python tests/golden/make_hand_closed_forms.py
"""
import json
import math
import os

e = math.e
ex = {
    "citation": ("Row layout: FlashInfer PR #4802 'Refactor Sparse MLA SM120', review note on "
                 "decode_dsv3_2_kernel.cuh (per-token KV layout: [0:512) e4m3, [512:528) 4 x fp32 "
                 "scale per 128-element tile, [528:656) 64 x bf16 rope). Sink/topk_length semantics: "
                 "vLLM PR #57673, Test Result section. The pages print no worked numbers; these values "
                 "are closed forms derived by hand from the definitions (softmax with an optional sink "
                 "logit added to the denominator only, natural-log LSE without the sink) and evaluated "
                 "with Python's math module."),
    "examples": [
        {
            "name": "two_rows_one_head",
            "derivation": ("row A: code 0x38 (=1.0) at nope[0], all scales 1.0; row B: code 0x40 (=2.0) "
                           "at nope[1], all scales 1.0; rope zero. q = e_0, sm_scale = 1. s_A = 1, s_B = 0. "
                           "out[0] = e/(e+1+S), out[1] = 2/(e+1+S) with S = exp(sink) (0 without sink); "
                           "lse = log(e+1)."),
            "H": 1, "sm_scale": 1.0,
            "rows": [{"codes": {"0": 0x38}, "scales": [1.0, 1.0, 1.0, 1.0], "rope": {}},
                     {"codes": {"1": 0x40}, "scales": [1.0, 1.0, 1.0, 1.0], "rope": {}}],
            "q": [{"0": 1.0}],
            "cases": [
                {"sink": None, "out": [{"0": e / (e + 1), "1": 2 / (e + 1)}], "lse": [math.log(e + 1)]},
                {"sink": [0.0], "out": [{"0": e / (e + 2), "1": 2 / (e + 2)}], "lse": [math.log(e + 1)]},
            ],
        },
        {
            "name": "scales_sign_rope_two_heads",
            "derivation": ("row A: code 0x38 (=1.0) at nope[0] with scale[0]=0.5, rope[0]=bf16 1.0 "
                           "(0x3F80); row B: code 0xB8 (=-1.0) at nope[0] with scale[0]=4, code 0x38 at "
                           "nope[200] with scale[1]=0.25, rope zero. Head 0: q=e_0; head 1: q=2*e_512 "
                           "(rope dim 0). sm_scale=1. Head 0: s_A=0.5, s_B=-4; head 1: s_A=2, s_B=0. "
                           "V_A=0.5 e_0; V_B=-4 e_0 + 0.25 e_200."),
            "H": 2, "sm_scale": 1.0,
            "rows": [{"codes": {"0": 0x38}, "scales": [0.5, 1.0, 1.0, 1.0], "rope": {"0": 0x3F80}},
                     {"codes": {"0": 0xB8, "200": 0x38}, "scales": [4.0, 0.25, 1.0, 1.0], "rope": {}}],
            "q": [{"0": 1.0}, {"512": 2.0}],
            "cases": [],
        },
    ],
}
a, b = math.exp(0.5), math.exp(-4)
c = math.exp(2)
for sink in (None, [1.0, -2.0]):
    s0 = 0.0 if sink is None else math.exp(sink[0])
    s1 = 0.0 if sink is None else math.exp(sink[1])
    ex["examples"][1]["cases"].append({
        "sink": sink,
        "out": [{"0": (0.5 * a - 4 * b) / (a + b + s0), "200": 0.25 * b / (a + b + s0)},
                {"0": (0.5 * c - 4) / (c + 1 + s1), "200": 0.25 / (c + 1 + s1)}],
        "lse": [math.log(a + b), math.log(c + 1)],
    })

here = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(here, "hand_closed_forms.json"), "w") as f:
    json.dump(ex, f, indent=1)
