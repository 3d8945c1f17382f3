"""Per-configuration table of the parity errors a GPU test session recorded.

    NF_PARITY_LOG=parity.json python -m pytest tests -m gpu -q
    python tests/parity_table.py parity.json > table.md

For each configuration (a set of tests and outputs), the worst over its checks
of the GPU output against the exact float64 oracle, against the bf16-storage
oracle, and of the storage term itself (bf16-storage against exact, computed
by the oracle alone).  Reads only the log; imports nothing of the library.
"""
import json
import re
import sys

# (label, output column, test name pattern, check name pattern)
CONFIGS = [
    ("small layer, all 35 two-way splits x 2 executors", "y", r"test_tiny_every_two_way_split$", r"^y$"),
    ("small layer", "appended k", r"test_tiny_every_two_way_split$", r"^appended k$"),
    ("small layer, attention output (intermediate)", "o", r"test_tiny_intermediates", r"^o$"),
    ("small layer, SwiGLU product (intermediate)", "a", r"test_tiny_intermediates", r"^a$"),
    ("small layer, prefill chunks after prefixes", "y", r"test_prefill_with_prefix", r"^y$"),
    ("degenerate batches (1 token, full block tables, page edges)", "y", r"test_degenerate_batches",
     r"^degenerate batch .*executor \d$"),
    ("small MoE layer, 4 plans", "y", r"test_tiny_moe_layer", r"^tiny MoE y$"),
    ("8B-shaped step, n = 1-4, sampled rows", "y", r"test_llama8b_sampled_rows_by_nano_batch_count",
     r"^y$"),
    ("8B-shaped step", "appended k", r"test_llama8b_sampled_rows_by_nano_batch_count",
     r"^appended k$"),
    ("8B shape, decode batches of 17-256 tokens", "y", r"test_llama8b_small_decode_batches", r"^y$"),
    ("3 small layers, both executors", "y", r"test_tiny_layers_step_matches_oracle", r"^3 tiny layers$"),
    ("small 3-layer stack", "logits", r"test_tiny_stack_matches_oracle", r"^3-layer tiny stack logits$"),
    ("8B-shaped 2-layer stack + LM head", "logits", r"test_llama8b_shaped_two_layer_stack",
     r"^8B-shaped 2-layer stack logits$"),
    ("8B-shaped decode-only batch (256 rows), 2 layers on one stream, 1 and 2 nano-batches", "y",
     r"test_llama8b_shaped_decode_layers_on_one_stream", r"^8B-shaped decode layers on one stream"),
    ("70B-shaped layer, sampled rows", "y", r"test_llama70b_shaped_layer_sampled_rows",
     r"^70B-shaped layer y$"),
    ("70B-shaped 2 layers, window n = 2 on 46 SMs", "y", r"test_llama70b_shaped_layers_overlapped",
     r"window n=2$"),
    ("70B-shaped 2 layers, window n = 3 on 45 SMs", "y", r"test_llama70b_shaped_layers_overlapped",
     r"window n=3$"),
    ("Mixtral-shaped MoE layer, sampled rows", "y", r"test_mixtral_shaped_layer_sampled_rows",
     r"^Mixtral-shaped y, bounds \[[0-9, ]*\]$"),
    ("runtime serving a random-weight 2-layer model, every iteration", "served logits",
     r"test_runtime_serves_a_real_model", r"^served logits, iteration \d+$"),
]


def table(entries):
    rows = ["| configuration | output | elements | exact oracle: max-abs / rel-L2 | "
            "bf16-storage oracle: max-abs / rel-L2 | storage term: max-abs / rel-L2 | rms(ref) |",
            "|---|---|---|---|---|---|---|"]
    for label, out, tpat, npat in CONFIGS:
        worst = {}
        n = {}
        rms = 0.0
        for e in entries:
            test = e["test"].split("::")[-1].split("[")[0]
            if not re.search(tpat, test):
                continue
            name = e["name"]
            storage = name.endswith(" (storage term)")
            base = name[: -len(" (storage term)")] if storage else name
            if not re.search(npat, base):
                continue
            kind = "storage" if storage else e["oracle"]
            w = worst.setdefault(kind, [0.0, 0.0])
            w[0] = max(w[0], e["max_abs"])
            w[1] = max(w[1], e["rel_l2"])
            if kind == "exact":
                n[label] = max(n.get(label, 0), e["n"])
                rms = max(rms, e["rms_ref"])
        if not worst:
            continue

        def cell(k):
            return f"{worst[k][0]:.4f} / {worst[k][1]:.2e}" if k in worst else "-"
        rows.append(f"| {label} | {out} | {n.get(label, 0)} | {cell('exact')} | "
                    f"{cell('bf16-storage')} | {cell('storage')} | {rms:.2f} |")
    return "\n".join(rows)


if __name__ == "__main__":
    print(table(json.load(open(sys.argv[1]))))
