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


def test_oracle_sample_is_the_oracle_forward():
    """The bench's timed CPU sample computes the oracle's stack forward of its rows and
    leading segments, with the weights taken from the host stack or drawn afresh."""
    import numpy as np
    from oracle import stack as S
    for cfg in (synth.MOE.with_(n_segments=4, tokens=12, hidden=16, ffn=8, n_experts=6, top_k=2),
                synth.DIT.with_(n_segments=3, tokens=10, hidden=16, ffn=24)):
        hs = synth.HostStack(cfg)
        for src in (hs, None):
            run = bench.OracleRun(cfg, 7, layers=2, hs=src)
            assert run.scale == cfg.n_segments / 2
            assert run.time_pass() > 0
            # the forward it times, replayed outside the timer
            x = run.x0
            F = run.F
            for s in range(2):
                if s in run.moe:
                    logits, experts = run._prepare(s)
                    x = F.moe_swiglu(x, logits, experts.__getitem__, cfg.top_k)
                else:
                    x = S.apply_segment(cfg, s, x, rows=run.rows, tensors=run._prepare(s))
            ref = S.stack_forward(cfg, rows=np.arange(7), n_segments=2)
            np.testing.assert_allclose(x, ref, rtol=1e-12, atol=1e-12)
            assert f"time scaled by {cfg.n_segments / 2:g}" in run.describe()


def test_traffic_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    import json
    from host_offloaded_weight_gb300 import profiling as P
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(P, "TRAFFIC_FILE", str(path))
    assert P.traffic("w", "gemm_up") is None                       # no capture
    entry = {"workload": "w", "kernel": "gemm_up", "dram_bytes_per_launch": 1234, "launches": 2,
             "source": P.SOURCES["gemm_up"], "source_sha256": P.source_sha("gemm_up"), "report": "r"}
    path.write_text(json.dumps({"entries": [entry]}))
    assert P.traffic("w", "gemm_up") == 1234
    assert P.traffic("w", "gemm_down") is None
    entry["source_sha256"] = "0" * 64                               # taken on another version
    path.write_text(json.dumps({"entries": [entry]}))
    assert P.traffic("w", "gemm_up") is None
