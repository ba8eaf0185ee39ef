"""The benchmark's roofline model (algorithmic bytes and FLOPs per call)
against per-token figures worked out by hand from the tensors a call must
touch. CPU only; nothing is launched."""
import bench
import workloads


def _per_token_head_bytes(name):
    wl = workloads.WORKLOADS[name]
    has_s0 = wl.s0
    total = bench.algorithmic_bytes(wl, has_s0)
    W = wl.dv + 1 if wl.mode == "elu1" else wl.dv
    state = 4 * wl.dk * W * (2 if has_s0 else 1)
    return (total / (wl.B * wl.H) - state) / wl.T


def test_bytes_per_token_and_head():
    # bf16 q, k, v read and o written: 2 * (128 + 128 + 128) + 2 * 128 = 1024 bytes at d = 128
    assert _per_token_head_bytes("retnet") == 1024
    # Gated DeltaNet adds a float32 gate and beta per token
    assert _per_token_head_bytes("gdn") == 1024 + 8
    # GLA adds a float32 gate per key channel; the outer-product gate one per value column too
    assert _per_token_head_bytes("gla") == 1024 + 4 * 128
    assert _per_token_head_bytes("outer") == 1024 + 4 * 128 + 4 * 128
    # elu+1 at d = 64: 2 * 64 * 4 bytes
    assert _per_token_head_bytes("elu1") == 512


def test_flops_per_token_and_head():
    C, d = 64, 128
    # unit write: scores 2 C dk, local output 2 C dv, inter-chunk output and state update 2 dk dv each
    assert bench.flops_per_token_head("retnet", d, d) == 2 * C * (d + d) + 4 * d * d
    # delta rule: K K^T, the WY products and the S-dependent correction on top, plus the C^2/3 solve
    assert bench.flops_per_token_head("gdn", d, d) == 2 * C * (3 * d + 2 * d) + C * C / 3.0 + 6 * d * d
    # the non-causal form has no scores: K^T V and Q S
    assert bench.flops_per_token_head("noncausal", d, d) == 4 * d * d


def test_backward_bytes_count_each_tensor_once():
    wl = workloads.WORKLOADS["backward"]
    per_head = bench.backward_bytes(wl) / (wl.B * wl.H)
    # q, k, v, dO read and dq, dk, dv written once (bf16), dS_final read and dS0 written once (float32)
    assert per_head == wl.T * 2 * (4 * 128 + 3 * 128) + 2 * 4 * 128 * 128
    wg = workloads.WORKLOADS["backward_gla"]
    # GLA also reads g and writes dg, both float32 per key channel
    assert bench.backward_bytes(wg) / (wg.B * wg.H) == per_head + wg.T * 8 * 128


def test_delta_rule_backward_bytes():
    # Gated DeltaNet: q, k, v, dO read and dq, dk, dv written (bf16); g and beta read, dg and dbeta
    # written (float32 per token); S0 and dS_final read and dS0 written (float32)
    wl = workloads.WORKLOADS["backward_gdn"]
    tok = 2 * (4 * 128 + 3 * 128) + 16
    assert bench.backward_bytes(wl) == wl.B * wl.H * (wl.T * tok + 3 * 4 * 128 * 128)
    # Kimi Delta Attention: the gate and its gradient per key channel instead of per token
    wk = workloads.WORKLOADS["backward_kda"]
    tok_k = 2 * (4 * 128 + 3 * 128) + 8 * 128 + 8
    assert bench.backward_bytes(wk) == wk.B * wk.H * (wk.T * tok_k + 3 * 4 * 128 * 128)


def test_kernel_sources_cover_every_workload_with_a_traffic_record():
    # every traffic record names a workload whose kernels' sources are listed, so that
    # the record's hash can be checked against them
    import re
    with open(bench.PROFILE_FILE) as f:
        names = re.findall(r"^traffic workload=(\S+)", f.read(), flags=re.M)
    assert names
    for n in names:
        assert n in bench.KERNEL_SOURCES, n


def test_kernel_names_follow_the_library_choice(monkeypatch):
    # the materialised variant of elu+1 (any B*H) takes the parallel state pass unless
    # LA_MAT_STATE=serial; RetNet's materialised pass stays serial; the delta rule and KDA
    # name their own kernels
    elu = workloads.WORKLOADS["elu1"]
    assert bench.kernel_name(elu) == "nc_sum_kernel+mat_scan_kernel+chunk_output_kernel"
    monkeypatch.setenv("LA_MAT_STATE", "serial")
    assert bench.kernel_name(elu) == "chunk_state_kernel+chunk_output_kernel"
    monkeypatch.delenv("LA_MAT_STATE")
    assert bench.kernel_name(workloads.WORKLOADS["gdn"]) == "chunk_delta_pair_kernel"
    assert bench.kernel_name(workloads.WORKLOADS["kda"]) == "kdw_pre_kernel+kdw_chain_kernel"
    small_retnet = workloads.WORKLOADS["retnet"].with_sizes(B=1, H=8, T=4096)
    assert bench.kernel_name(small_retnet).startswith("chunk_state_kernel+")
    assert not bench.parallel_state_pass(small_retnet)
