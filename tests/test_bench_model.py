"""The bench's per-launch FLOP and byte model against hand counts, and its reference arm (no GPU)."""
import bench
import synth

RIDGE = 1943.5e12 / 6760.6e9      # measured bf16 FLOP/s over measured HBM bytes/s


def test_dit_counts_by_hand():
    cfg = synth.STACKS["dit_ffn_12x1024x4096"]
    T, H, F = 4096, 1024, 4096
    kf, kb = bench.kernel_flops(cfg, T), bench.kernel_bytes(cfg, T)
    assert kf["gemm_up"] == kf["gemm_down"] == 2 * T * H * F == 34_359_738_368
    # x, W1, b1 in; H out (bf16)
    assert kb["gemm_up"] == 2 * (T * H + F * H + F + T * F) == 50_339_840
    # H, W2, b2 in, fp32 residual in; bf16 and fp32 out
    assert kb["gemm_down"] == 2 * (T * F + H * F + H) + 4 * T * H + 2 * T * H + 4 * T * H
    assert kf["gemm_up"] / kb["gemm_up"] > RIDGE and kf["gemm_down"] / kb["gemm_down"] > RIDGE


def test_swiglu_counts_both_matrices():
    cfg = synth.STACKS["swiglu_48x5120x13824"]
    T, H, F = cfg.tokens, cfg.hidden, cfg.ffn
    kf, kb = bench.kernel_flops(cfg, T), bench.kernel_bytes(cfg, T)
    assert kf["gemm_up"] == 2 * kf["gemm_down"] == 4 * T * H * F
    assert kb["gemm_up"] == 2 * T * H + 2 * (2 * F * H) + 2 * F + 2 * T * F
    assert "gemm_proj" not in kb


def test_moe_expert_gemms_sit_below_the_ridge():
    cfg = synth.STACKS["moe_48x128x2048x768"]
    T, H, F, k, E = cfg.tokens, cfg.hidden, cfg.ffn, cfg.top_k, cfg.n_experts
    kf = bench.kernel_flops(cfg, T)
    kb_all = bench.kernel_bytes(cfg, T)
    assert kb_all["gemm_up"] == 2 * (T * k * H + E * 2 * F * H + T * k * F)
    assert kb_all["gemm_down"] == 2 * (T * k * F + E * H * F) + 4 * T * k * H
    # every expert's weights are read once per layer: ~100 FLOP per byte, HBM-bound
    for name in ("gemm_up", "gemm_down"):
        assert kf[name] / kb_all[name] < RIDGE / 2
    # fewer routed experts move fewer weight bytes; the row traffic stays
    kb_half = bench.kernel_bytes(cfg, T, routed=E / 2)
    assert kb_all["gemm_up"] - kb_half["gemm_up"] == 2 * (E / 2) * 2 * F * H


def test_reference_arm_line():
    """`bench.py --impl reference` on the host: one JSON line with the contract's keys, the
    oracle as the timed program, the line's own value as its cpu_baseline and e2e."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--ref-tokens", "8", "--workload", "tiny_f32_4x256"],
                         cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_f32_4x256"
