"""Named synthetic decode workloads (shapes, dtypes, sparsity profiles).

Each entry describes the seeded synthetic input of one FFN decode workload;
``synth.make_layer`` / ``synth.gen_x`` turn it into bytes.  The activation
profile is a Zipf curve p_i = min(0.9, c * (i+1)^-alpha) over hot-first
neuron order, with c calibrated so that the mean of p_i equals the stated
density (``literal_c`` keeps a printed constant instead, as a variant).
"""
from __future__ import annotations

WORKLOADS = {
    # tiny single ReLU FFN layer
    "relu_ffn_d1024_n4096_r64_f16": dict(
        d=1024, n=4096, r=64, dtype="f16", gated=False, alpha=0.8, density=0.08,
        literal_c=0.5, seed=1, steps=64, layers=1, batch=1),
    # OPT-6.7B-shaped single FFN
    "opt6.7b_ffn_d4096_n16384_r128_f16": dict(
        d=4096, n=16384, r=128, dtype="f16", gated=False, alpha=0.9, density=0.06,
        seed=2, steps=256, layers=1, batch=1),
    # ReLU-fied Llama-2-7B-shaped gated FFN
    "llama2_7b_gated_ffn_d4096_n11008_r256_bf16": dict(
        d=4096, n=11008, r=256, dtype="bf16", gated=True, alpha=1.0, density=0.10,
        seed=3, steps=64, layers=1, batch=1),
    # OPT-30B-shaped 48-layer FFN stack with residual adds
    "opt30b_ffn_stack_48x_d7168_n28672_r256_f16": dict(
        d=7168, n=28672, r=256, dtype="f16", gated=False, alpha_range=(0.7, 1.2),
        density_range=(0.15, 0.03), seed=4, steps=128, layers=48, batch=1),
    # OPT-13B-shaped batched decode and density sweep
    "opt13b_ffn_batched_d5120_n20480_r192_f16": dict(
        d=5120, n=20480, r=192, dtype="f16", gated=False, alpha=0.9,
        densities=(0.02, 0.05, 0.10, 0.25, 0.50), batches=(1, 4, 16, 32),
        seed=5, steps=32, layers=1),
}

TINY = "relu_ffn_d1024_n4096_r64_f16"
OPT67 = "opt6.7b_ffn_d4096_n16384_r128_f16"
LLAMA_GATED = "llama2_7b_gated_ffn_d4096_n11008_r256_bf16"
OPT30_STACK = "opt30b_ffn_stack_48x_d7168_n28672_r256_f16"
OPT13_BATCHED = "opt13b_ffn_batched_d5120_n20480_r192_f16"
