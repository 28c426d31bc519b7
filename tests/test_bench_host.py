"""Host-side arithmetic of bench.py: the algorithmic bytes and flops the
roofline fractions divide by, against their closed forms at the benchmarked
shape (4 requests x 512 beams, 16 query / 8 kv heads, head_dim 128, prompts
of 4096, bf16 KV, vocab 151936, last of 3 decode steps)."""
import bench
import synth


def test_algorithmic_units_of_the_benchmarked_step():
    wl = synth.WORKLOADS["onerec17b"]
    rows = wl.R * wl.W                                                 # 2048 live beams
    assert bench.algorithmic(wl, rows, "bd_stream_select_kernel") == (2048 * 151936 * 4, "bytes")
    flops, kind = bench.algorithmic(wl, rows, "bd_attn_shared_tc_kernel")
    # 4 (QK^T and PV, 2 flops per MAC) x kv heads x (W x G) rows x sum P keys x d
    assert kind == "flops" and flops == 4 * 8 * (512 * 2) * (4 * 4096) * 128 == 68719476736


def test_algorithmic_units_of_the_open_vocabulary_selection():
    wl = synth.WORKLOADS["openvocab"]
    rows = wl.R * wl.W                                                 # 10000 live beams
    # the expansion kernel reads every live logits row in full, like the normaliser stream
    assert bench.algorithmic(wl, rows, "bd_expand_kernel") == (10000 * 151936 * 4, "bytes")
    assert bench.algorithmic(wl, rows, "bd_stream_select_kernel") == (10000 * 151936 * 4, "bytes")
    # with a trie the expansion reads only children windows: a bound of 2 x 4 B per kept candidate
    tr = synth.WORKLOADS["onerec17b"]
    assert bench.algorithmic(tr, 2048, "bd_expand_kernel") == (2048 * 2 * 4 * 512, "bytes")


def test_step_roofline_counts_prompt_kv_once_per_request():
    wl = synth.WORKLOADS["onerec17b"]
    kernels = {"bd_stream_select_kernel": {"us_per_launch": 200.0},
               "bd_attn_shared_tc_kernel": {"us_per_launch": 80.0}}
    out = bench.step_roofline(wl, 2048, 0.3, kernels, {})
    shared = 4 * 4096 * 8 * 128 * 2 * 2          # K and V of every prompt, bf16, once per request
    unshared = 2048 * 3 * 8 * 128 * 2 * 2        # 3 decode tokens per beam at the last step
    qo = 2 * 2048 * 16 * 128 * 2                 # queries in, outputs out, bf16
    assert out["attention"]["bytes"] == shared + unshared + qo == 109051904
    assert out["attn_select_bytes"] == shared + unshared + qo + 2048 * 151936 * 4
    assert abs(out["attn_select_gbs"] - out["attn_select_bytes"] / 0.3e-3 / 1e9) < 0.1
    assert out["attention"]["us"] == 80.0 and out["attention"]["binding"] == "tensor"
    # binding roof: the tensor time at the bf16 burst peak (the attention
    # kernels run alone for tens of microseconds); fallback 1.9 PFLOP/s here
    assert abs(out["attention"]["roof_us"]["tensor"] - 68719476736 / 1.9e15 * 1e6) < 0.01
    # the conservative denominator: distinct unshared rows instead of per-beam reads
    out2 = bench.step_roofline(wl, 2048, 0.3, kernels, {}, unique_slots=1000)
    assert out2["attention"]["bytes_unique_slots"] == shared + 1000 * 8 * 128 * 2 * 2 + qo


def test_workload_dtype_names_each_workloads_types():
    assert bench.workload_dtype(synth.WORKLOADS["onerec17b"]) == \
        "f32 logits; bf16 q / bf16 KV / bf16 out, f32 accumulate"
    assert bench.workload_dtype(synth.WORKLOADS["fp8kv"]).startswith("f32 logits; bf16 q / e4m3 KV")
    assert bench.workload_dtype(synth.WORKLOADS["tiny"]).startswith("f32 logits; f32 q / f32 KV")


def test_both_arms_name_the_workload_alike():
    wl = synth.WORKLOADS["onerec17b"]
    assert bench.workload_name(wl, wl.T - 1) == ("onerec17b: R4 P4096 Hq16 Hkv8 d128 W512 K512 V151936 "
                                                 "SID 3x8192 catalog 4000000 step 3/3")


def test_traffic_rows_count_only_for_their_workload_and_source(tmp_path, monkeypatch):
    import hashlib
    csrc = tmp_path / "wide_beam_generative_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "select.cu").write_text("// kernel source\n")
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()[:12]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        "| kernel | workload | bytes per launch | source sha256[:12] | capture |\n|---|---|---|---|---|\n"
        f"| bd_stream_select_kernel | onerec17b | 1234 | {sha} | x |\n"
        "| bd_stream_select_kernel | fp8kv | 99 | 000000000000 | stale source |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("bd_stream_select_kernel", "onerec17b") == 1234.0
    assert bench.read_traffic("bd_stream_select_kernel", "openvocab") is None   # no row for it
    assert bench.read_traffic("bd_stream_select_kernel", "fp8kv") is None       # taken on other source
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        "| kernel | workload | bytes per launch | source sha256[:12] | capture |\n|---|---|---|---|---|\n"
        f"| bd_seed_kernel | openvocab | 77 | {sha} | x |\n"
        f"| bd_unknown_kernel | openvocab | 88 | {sha} | x |\n")
    assert bench.read_traffic("bd_seed_kernel", "openvocab") == 77.0
    assert bench.read_traffic("bd_unknown_kernel", "openvocab") is None         # no source file known


def test_cpu_sample_is_bounded():
    """The oracle's timed sample stays at four requests' worth of rows,
    capped for the wide open-vocabulary rows."""
    assert bench.default_cpu_rows(synth.WORKLOADS["onerec17b"]) == 2048
    assert bench.default_cpu_rows(synth.WORKLOADS["qwen06b"]) == 200
    assert bench.default_cpu_rows(synth.WORKLOADS["openvocab"]) == 1024
