"""The committed ncu traffic figures: each entry matches the summary it cites,
and the DRAM bytes of a stage-1 launch stay within a few percent of the
algorithmic bytes (KV + q + out) of its workload, i.e. nothing is re-read."""
import json
import os

import workloads as synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KV_BYTES = {"bf16": 1152, "fp8": 576, "mxfp4": 288 + 18}


def algorithmic_bytes(name):
    c = synth.CONFIGS[name]
    lengths = synth.config_lengths(name)
    q = len(lengths) * 16 * 576 * (2 if c["q_dtype"] == "bf16" else 1)
    out = len(lengths) * 16 * 512 * 2
    return sum(lengths) * KV_BYTES[c["kv_dtype"]] + q + out


def test_traffic_entries_match_their_summaries_and_the_algorithmic_bytes():
    with open(os.path.join(ROOT, "profiles", "stage1_traffic.json")) as f:
        entries = {k: v for k, v in json.load(f).items() if not k.startswith("_")}
    assert entries
    for name, e in entries.items():
        summary = e["source"].split(":")[0]
        with open(os.path.join(ROOT, summary)) as f:
            text = f.read()
        assert e["stage1_sha"] in text, f"{summary} was not written for kernel {e['stage1_sha']}"
        ratio = e["dram_bytes_per_launch"] / algorithmic_bytes(name)
        assert 0.98 < ratio < 1.03, f"{name}: DRAM bytes / algorithmic bytes = {ratio:.4f}"
