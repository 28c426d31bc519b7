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
    # binding roof: the tensor time at the fallback sustained peak
    assert abs(out["attention"]["roof_us"]["tensor"] - 68719476736 / 1.7e15 * 1e6) < 0.01


def test_both_arms_name_the_workload_alike():
    wl = synth.WORKLOADS["onerec17b"]
    assert bench.workload_name(wl, wl.T - 1) == ("onerec17b: R4 P4096 Hq16 Hkv8 d128 W512 K512 V151936 "
                                                 "SID 3x8192 catalog 4000000 step 3/3")
