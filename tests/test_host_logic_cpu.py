"""Host-side logic that needs no GPU: the seeded input generators (the one
module the CUDA path and the oracle share), and the benchmark's bookkeeping
(which kernel a workload runs, when a committed ncu figure still applies,
the algorithmic byte counts)."""
import json
import os

import numpy as np
import pytest
import torch

import bench
from draft_verify_acceptance_gb300 import workloads as W


def test_inputs_are_a_function_of_the_seed():
    a = W.make_inputs(3, 2, 64, seed=5)
    b = W.make_inputs(3, 2, 64, seed=5)
    c = W.make_inputs(3, 2, 64, seed=6)
    for x, y in zip((a.target, a.draft, a.tokens, a.uniforms), (b.target, b.draft, b.tokens, b.uniforms)):
        assert torch.equal(x, y)
    assert not torch.equal(a.target, c.target)


def test_input_streams_are_independent():
    """Changing the draft noise changes neither the target logits nor the
    uniforms (one generator stream per input)."""
    a = W.make_inputs(4, 3, 100, seed=2, draft_noise=0.5)
    b = W.make_inputs(4, 3, 100, seed=2, draft_noise=2.0)
    assert torch.equal(a.target, b.target) and torch.equal(a.uniforms, b.uniforms)
    assert not torch.equal(a.draft, b.draft)


def test_draft_tokens_in_range_and_greedy_tokens_from_noisy_argmax():
    s = W.make_inputs(8, 4, 50, seed=1)
    assert s.tokens.dtype == torch.int32 and int(s.tokens.min()) >= 0 and int(s.tokens.max()) < 50
    g = W.make_inputs(8, 4, 50, seed=1, mode=W.MODE_GREEDY, greedy_noise=0.0)
    # with no noise the draft is the target's own argmax: every token accepted
    assert torch.equal(g.tokens.long(), g.target[:, :4].float().argmax(-1))
    assert g.draft is None and g.uniforms is None


def test_uniforms_in_unit_interval():
    u = W.make_inputs(64, 8, 10, seed=3).uniforms
    assert float(u.min()) >= 0.0 and float(u.max()) < 1.0


def test_scd_inputs_hold_the_amateur_at_every_position():
    inp = W.make_scd_inputs(4, 3, 64, seed=4, amateur_noise=0.25)
    assert inp.draft.shape == (4, 4, 64)  # K + 1 amateur rows
    d = (inp.draft - inp.target).float()
    assert 0.15 < float(d.std()) < 0.35
    ind = W.make_scd_inputs(4, 3, 64, seed=4, independent_amateur=True)
    assert abs(float(np.corrcoef(ind.draft.flatten(), ind.target.flatten())[0, 1])) < 0.1


def test_reward_scores_recipe():
    s = W.make_scores(64, 2000, seed=0)
    assert s.dtype == torch.float32 and s.shape == (64, 2000)
    mu, sd = s.double().mean(1), s.double().std(1)
    assert float(mu.std()) > 1.0  # prompts differ in their reward level
    assert float(sd.min()) > 0.2 and float(sd.max()) < 5.0
    t = W.make_scores(8, 500, kind="ties", seed=0)
    v = t.numpy()
    assert set(np.unique(v)) <= set(range(-3, 4))
    assert np.signbit(v[v == 0]).any() and (~np.signbit(v[v == 0])).any()  # both zeros
    with pytest.raises(ValueError):
        W.make_scores(2, 2, kind="other")


@pytest.mark.parametrize("name", list(W.WORKLOADS))
@pytest.mark.parametrize("B", [2, None, 152, 153, 400])
def test_kernel_plan_matches_the_dispatch_rule(name, B):
    """The bench's restatement of launch_sample's dispatch: at most one
    sequence per SM (152) whose 2K+1 rows fit 192 KiB -> the small-batch
    kernel; else rows of at most 4096 vectors -> the fused kernel; longer rows
    -> the two-kernel sampler."""
    import types
    spec = W.WORKLOADS[name]
    inp = types.SimpleNamespace(B=spec["B"] if B is None else B, K=spec["K"], V=spec["V"],
                                mode=spec["mode"],
                                dtype_name="bf16" if spec["dtype"] == torch.bfloat16 else "f32")
    kernel, launches = bench.kernel_plan(inp)
    if spec["mode"] == W.MODE_GREEDY:
        assert (kernel, launches) == ("greedy_kernel", 1)
    else:
        esz = 2 if spec["dtype"] == torch.bfloat16 else 4
        nvec = spec["V"] * esz // 16
        K = spec["K"]
        if inp.B <= 152 and (2 * K + 1) * nvec * 16 <= 192 * 1024:
            want = ("seq_sample_kernel", 1)
        elif nvec <= 4096:
            want = ("fused_sample_kernel", 1)
        else:
            want = ("norm_stream_kernel", 2)
        assert (kernel, launches) == want
    if name == "tiny_sample_f32_B4_K4_V1000" and inp.B <= 152:
        assert kernel == "seq_sample_kernel"
    if name == "best_of_n_bf16_B1024_K4_V32000":
        assert kernel == "fused_sample_kernel"


def test_algorithmic_bytes_count_every_row_once():
    inp = W.make_inputs(2, 3, 1000, seed=0)
    s = 4
    want = 2 * 4 * 1000 * s + 2 * 3 * 1000 * s + 2 * 3 * 4 + 2 * 4 * 4 + 2 * 4 + 2 * 4 * 4
    assert inp.algorithmic_bytes() == want
    g = W.make_inputs(2, 3, 1000, seed=0, mode=W.MODE_GREEDY)
    assert g.algorithmic_bytes() == 2 * 4 * 1000 * s + 2 * 3 * 4 + 2 * 4 + 2 * 4 * 4


def test_committed_traffic_applies_only_to_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for workload, e in d.items():
        if workload.startswith("_"):
            continue
        assert e["kernel"] in bench.KERNEL_SOURCES, workload
        assert e["dram_bytes_per_launch"] > 0
        assert bench.committed_traffic(workload, e["kernel"]) in (e["dram_bytes_per_launch"], None)
    # a different kernel name, or a changed source hash, gives no figure
    assert bench.committed_traffic("greedy_bf16_B64_K8_V32000", "fused_sample_kernel") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0000000000000000")
    assert bench.committed_traffic("greedy_bf16_B64_K8_V32000", "greedy_kernel") is None


def test_hbm_peak_falls_back_without_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, kind = bench.hbm_peak()
    assert kind == "fallback" and peak == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.5}))
    assert bench.hbm_peak() == (7000.5, "measured")


def test_kernel_hash_ignores_comments_only():
    src = 'int f() { return 1; } // note\n/* block\n comment */ const char* s = "// kept";\n'
    assert bench.strip_comments(src) == 'int f() { return 1; } \n  const char* s = "// kept";\n'
    files = {f: "" for f in bench.KERNEL_SOURCES["greedy_kernel"]}
    files["verify_greedy.cu"] = "int x = 1; // one\n"
    h0 = bench.kernel_source_hash("greedy_kernel", files.get)
    files["verify_greedy.cu"] = "int x = 1; /* the same code */ // another comment\n"
    h1 = bench.kernel_source_hash("greedy_kernel", files.get)
    files["verify_greedy.cu"] = "int x = 2; // one\n"
    h2 = bench.kernel_source_hash("greedy_kernel", files.get)
    assert h0 == h1 != h2


def test_early_exit_schedule_matches_the_dispatch_rule():
    """The bench's restatement of the early-exit dispatch: rows whose two
    slices (and lane checkpoints) fit 200 KiB in a cluster of at most 8 CTAs
    take the cluster kernel; longer rows the two-phase schedule; small
    batches that fit one CTA per sequence the small-batch kernel."""
    import types
    # cluster sizes at the bench's vocabularies and at the limits
    assert bench.ee_cluster_size(32000 * 2 // 16) == 1
    assert bench.ee_cluster_size(20000 * 4 // 16) == 1
    assert bench.ee_cluster_size(65536 * 2 // 16) == 2
    assert bench.ee_cluster_size(128256 * 2 // 16) == 4
    assert bench.ee_cluster_size(152064 * 4 // 16) == 8
    assert bench.ee_cluster_size(400000 * 2 // 16) == 0
    nv = 6144  # a slice of 6144 vectors: 192 KiB of rows + 6 checkpoint groups > 200 KiB
    assert bench.ee_cluster_size(8 * nv) == 0 and bench.ee_cluster_size(8 * 6000) == 8
    want = {"tiny_sample_f32_B4_K4_V1000": "small_batch"}
    for name, spec in W.WORKLOADS.items():
        if spec["mode"] != W.MODE_SAMPLE or spec["K"] == 0:
            continue
        inp = types.SimpleNamespace(B=spec["B"], K=spec["K"], V=spec["V"],
                                    target=torch.empty(0, dtype=spec["dtype"]))
        assert bench.early_exit_schedule(inp) == want.get(name, "cluster"), name
    inp = types.SimpleNamespace(B=4, K=2, V=400000, target=torch.empty(0, dtype=torch.bfloat16))
    assert bench.early_exit_schedule(inp) == "two_phase"
