"""Writes oracle_ar_streams.txt: the CPU oracle's own greedy AR tokens after each bench workload's
prompt, the reference tokens of the seeded drafts when the oracle itself is timed (bench.py's
cpu_baseline and --impl reference legs), so that no input of the oracle comes from the GPU.

Calls only the oracle (oracle/) and the seeded input generators (spd_inputs).  Workloads that share
the target model and prompt (the 9B-class model at n = 4, 8, 16) share one stream.

    python tests/golden/make_oracle_ar.py [count]
"""
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import spd_inputs as si  # noqa: E402
from oracle import model as om  # noqa: E402

OUT = os.path.join(HERE, "oracle_ar_streams.txt")
WORKLOADS = ("dense1.5b_bf16_n8", "gqa4b_bf16_n8", "gqa9b_bf16_n8")


def target_names(w):
    return [n for n, _, _ in si.weight_specs(w) if not n.startswith("pdm.")]


def main(count: int) -> None:
    lines = ["# CPU oracle greedy AR after each workload's prompt (fp32 numpy, oracle/model.py greedy_ar)",
             "# written by tests/golden/make_oracle_ar.py; columns: workload prompt_len count tokens at P+1..P+count"]
    for name in WORKLOADS:
        w = si.WORKLOADS[name]
        t0 = time.time()
        params = si.generate_weights(w, device="cpu", names=target_names(w))
        target = om.Decoder(w.model, params)
        del params
        prompt = si.prompt_tokens(w).tolist()
        toks = om.greedy_ar(target, prompt, count)["tokens"]
        del target
        lines.append(" ".join([name, str(len(prompt)), str(count)] + [str(t) for t in toks]))
        print(f"{name}: {count} tokens in {time.time() - t0:.0f} s", flush=True)
    with open(OUT, "w") as fh:
        fh.write("\n".join(lines) + "\n")


def load():
    """{workload: (prompt_len, tokens)} from the stored file."""
    out = {}
    with open(OUT) as fh:
        for ln in fh:
            if ln.startswith("#") or not ln.strip():
                continue
            f = ln.split()
            out[f[0]] = (int(f[1]), [int(x) for x in f[3:3 + int(f[2])]])
    return out


def stream_for(w):
    """The stored stream of workload `w`, or of a stored workload with the same model and prompt."""
    table = load()
    for name, (plen, toks) in table.items():
        s = si.WORKLOADS[name]
        if (s.model, s.weight_seed, s.prompt_seed, s.prompt_len) == (w.model, w.weight_seed, w.prompt_seed,
                                                                     w.prompt_len):
            return toks
    return None


if __name__ == "__main__":
    main(int(sys.argv[1]) if len(sys.argv) > 1 else 128)
