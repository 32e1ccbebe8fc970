"""Write tests/golden/seeds.json: per workload, the query re-draw of each prompt
whose oracle chunk scores leave a safe cut-off margin (see margins.py).

Calls only the synthetic-input generators and the float64 oracle. Run from
the repository root:  python -m tests.golden.make_seeds [workload ...]
"""

import json
import os
import sys
import time

import numpy as np

import oracle
from synth import WORKLOADS, make_inputs
from synth.inputs import background_keys, prompt_lengths
from tests.golden.margins import CROSSING_GAP, RANK_GAP, margins_ok, prompt_margins

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "seeds.json")
MAX_ATTEMPTS = 200


def search(name: str) -> dict:
    w = WORKLOADS[name]
    lengths = prompt_lengths(w)
    kb = background_keys(w, lengths)
    attempts = [0] * len(lengths)
    pending = list(range(len(lengths)))
    per_prompt = [None] * len(lengths)
    tries = 0
    while pending:
        inp = make_inputs(w, prompt_attempts=attempts, k_background=kb)
        out = oracle.run(inp.q, inp.k, inp.seq_off, **w.selection_kwargs())
        coff = out["chunk_off"]
        still = []
        for b in pending:
            m = prompt_margins(out["chunk_score"][coff[b]:coff[b + 1]], w.mode, w.keep_p, w.mass)
            if margins_ok(m):
                per_prompt[b] = m
            else:
                attempts[b] += 1
                still.append(b)
        pending = still
        tries += 1
        if tries > MAX_ATTEMPTS:
            raise RuntimeError(f"{name}: no margin after {MAX_ATTEMPTS} re-draws")
    kept = int(out["kept_off"][-1])
    return {
        "prompt_attempts": attempts,
        "lengths": [int(v) for v in lengths],
        "margins": per_prompt,
        "kept_tokens": kept,
        "kept_fraction": kept / float(inp.n_tokens_total),
        "ranked_chunks": int((out["chunk_keep"] & 1).sum()),
        "rounds": tries,
    }


def main(names):
    table = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            table = json.load(f)
    table["_rule"] = {"rank_gap": RANK_GAP, "crossing_gap": CROSSING_GAP,
                      "how": "first query re-draw per prompt meeting both margins on oracle scores"}
    for name in names:
        t0 = time.time()
        table[name] = search(name)
        print(name, table[name]["prompt_attempts"], f"{time.time() - t0:.1f}s", flush=True)
        with open(OUT, "w") as f:
            json.dump(table, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or [n for n in WORKLOADS])
