"""Write the oracle regression fixtures in this folder.

The pages print no worked numeric example for the attention forward (the
fuel-dispatch contracts and the gfx942 derivation give definitions and a
tolerance, never an input with its output), so the fixtures here are small
seeded problems whose expected outputs come from the float64 oracle alone.
They pin the oracle across machines and compilers (x86_64 here, aarch64 next
to the GPU): a later change to the oracle that moves any value fails
tests/test_golden.py.

Run:  python tests/golden/make_golden.py
Calls only the oracle package and the seeded input generator.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import torch  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

CASES = [
    dict(name="mha_noncausal_f32", B=1, Hq=2, Hkv=2, Sq=5, Sk=6, D=4, dtype="f32",
         causal=False, wl=None, wr=None, softcap=None, alibi=False, empty=0.0,
         cite="attention.fkc.md, attention_naive: scale, stable softmax, weighted V sum"),
    dict(name="gqa_causal_bf16", B=2, Hq=4, Hkv=2, Sq=6, Sk=6, D=8, dtype="bf16",
         causal=True, wl=None, wr=None, softcap=None, alibi=False, empty=0.0,
         cite="attention.fkc.md, header: GQA broadcast of kv head h / (Hq/Hkv); position_admissible (causal)"),
    dict(name="window_softcap_alibi_bf16", B=1, Hq=2, Hkv=1, Sq=9, Sk=9, D=4, dtype="bf16",
         causal=True, wl=3, wr=0, softcap=2.0, alibi=True, empty=0.2,
         cite="attention.fkc.md, attention_naive: softcap tanh(s/c)*c, then ALiBi slope*(kj-qi); window; fully-masked row -> zeros"),
]

# Backward by recompute (attention.fkc.md, attention_flash_backward): dQ, dK, dV
# for a seeded dO, expected values from oracle.attn_bwd alone.
BWD_CASES = [
    dict(name="bwd_gqa_causal_bf16", B=1, Hq=4, Hkv=2, Sq=7, Sk=7, D=8, dtype="bf16",
         causal=True, wl=None, wr=None, softcap=None, alibi=False, empty=0.0,
         cite="attention.fkc.md, attention_flash_backward: recompute P, dV, dP, dS, dQ, dK; GQA sums"),
    dict(name="bwd_window_softcap_alibi_f32", B=1, Hq=2, Hkv=1, Sq=8, Sk=9, D=4, dtype="f32",
         causal=True, wl=3, wr=None, softcap=2.0, alibi=True, empty=0.25,
         cite="attention.fkc.md, attention_flash_backward: softcap factor 1 - tanh^2(s_pre/c); "
              "a fully-masked row contributes nothing"),
]

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def inputs(c):
    dt = DT[c["dtype"]]
    q = synth.normal((c["B"], c["Hq"], c["Sq"], c["D"]), 7, synth.STREAM_Q, dt)
    k = synth.normal((c["B"], c["Hkv"], c["Sk"], c["D"]), 7, synth.STREAM_K, dt)
    v = synth.normal((c["B"], c["Hkv"], c["Sk"], c["D"]), 7, synth.STREAM_V, dt)
    slopes = synth.alibi_slopes(c["Hq"]) if c["alibi"] else None
    rb = None
    if c["empty"]:
        rb = synth.row_kv_bounds_with_empty_rows(c["B"], c["Sq"], c["Sk"], c["empty"], seed=7)
    return q, k, v, slopes, rb


def run(c):
    q, k, v, slopes, rb = inputs(c)
    return oracle.attn(q, k, v, causal=c["causal"], window_left=c["wl"], window_right=c["wr"],
                       softcap=c["softcap"], alibi_slopes=slopes, row_kv_bounds=rb, return_lse=True)


def run_bwd(c):
    q, k, v, slopes, rb = inputs(c)
    do = synth.normal((c["B"], c["Hq"], c["Sq"], c["D"]), 7, synth.STREAM_DO, DT[c["dtype"]])
    return oracle.attn_bwd(q, k, v, do, causal=c["causal"], window_left=c["wl"], window_right=c["wr"],
                           softcap=c["softcap"], alibi_slopes=slopes, row_kv_bounds=rb)


def main():
    for c in BWD_CASES:
        rec = dict(c)
        for name, t in zip(("dq", "dk", "dv"), run_bwd(c)):
            rec[name] = [float.hex(x) for x in t.reshape(-1).tolist()]
        with open(os.path.join(HERE, c["name"] + ".json"), "w") as f:
            json.dump(rec, f, indent=0)
            f.write("\n")
    for c in CASES:
        out, lse = run(c)
        rec = dict(c)
        rec["out"] = [float.hex(x) for x in out.view(-1).tolist()]
        rec["lse"] = [float.hex(x) for x in lse.view(-1).tolist()]
        with open(os.path.join(HERE, c["name"] + ".json"), "w") as f:
            json.dump(rec, f, indent=0)
            f.write("\n")


if __name__ == "__main__":
    main()
