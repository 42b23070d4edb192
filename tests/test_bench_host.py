"""Host-side pieces of bench.py: the byte model behind every GB/s figure, the
CPU-baseline samples and the recorded-traffic lookup (no GPU needed)."""
import os

import pytest
import torch

import bench
import workloads as W


def test_byte_model_of_the_hot_path_workloads():
    """Read + write of the rotated elements, plus cos/sin (or one gathered cache
    row per token) and the positions, worked out from the shapes by hand."""
    inplace, neox, gptj, mrope = bench.build_workloads()
    # x bf16 [4,4096,32,128], slice of 64: read+write; cos/sin f32 [1,4096,1,64] read
    assert bench.algorithmic_bytes(inplace) == 4 * 4096 * 32 * 64 * 2 * 2 + 2 * 4096 * 64 * 4 == 136314880
    # q 32 + k 8 heads of 128 bf16 read+write per token, one 128-wide cache row, one int64 position
    assert bench.algorithmic_bytes(neox) == 16384 * (40 * 128 * 2 * 2 + 128 * 2 + 8) == 339869696
    # 16 + 16 heads, only R = 64 of 256 columns touched, f16
    assert bench.algorithmic_bytes(gptj) == 8192 * (32 * 64 * 2 * 2 + 64 * 2 + 8) == 68222976
    # 28 + 4 heads of 128 bf16, one cache row-equivalent, three int64 positions
    assert bench.algorithmic_bytes(mrope) == 32768 * (32 * 128 * 2 * 2 + 128 * 2 + 3 * 8) == 546045952
    small = W.inplace_f32_small("slice")  # x f32 [1,16,2,64], slice [16,48): 32 columns
    assert bench.algorithmic_bytes(small) == 16 * 2 * 32 * 4 * 2 + 2 * 16 * 32 * 4 == 12288


def test_byte_model_of_the_fused_op():
    c = W.qkv_case("bytes", 1, [5, 1, 3], [0, 7, 20], 4, 2, 2, 64, 4, torch.bfloat16, pad_every=4)
    T, D, e = 9, 64, 2
    cached = int((c.slot_mapping >= 0).sum())
    assert cached < T  # padding slots write no cache rows
    want = (T * 8 * D * e            # qkv read
            + T * 4 * D * e          # q_out written
            + cached * 4 * D * e     # k and v rows cached
            + T * D * e              # one cos/sin row per token
            + 2 * D * e              # the two gammas
            + (3 + 4 + 9) * 8)       # seqLens, queryStartLoc, slotMapping
    assert bench.algorithmic_bytes(c) == want


def test_cpu_samples_cover_whole_batches_and_prefixes():
    inplace, neox, gptj, mrope = bench.build_workloads()
    whole = bench.oracle_sample(inplace, inplace.tokens)
    assert tuple(whole.x.shape) == (4, 4096, 32, 128)
    assert bench.algorithmic_bytes(whole) == bench.algorithmic_bytes(inplace)
    assert tuple(bench.oracle_sample(inplace, 5000).x.shape) == (1, 4096, 32, 128)
    part = bench.oracle_sample(inplace, 300)
    assert tuple(part.x.shape) == (1, 300, 32, 128) and tuple(part.cos.shape) == (1, 300, 1, 64)
    m = bench.oracle_sample(mrope, 1000)
    assert m.tokens == 1000 and tuple(m.positions.shape) == (3, 1000)
    assert torch.equal(m.query, mrope.query[:1000])


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    label = "mrope_neox_bf16_32768tok_28q4k_h128_s16_24_24"
    (tmp_path / "profiles").mkdir()
    table = tmp_path / "profiles" / "dram_traffic.txt"
    table.write_text("kernel_source_sha256_16: %s\n%s: 123456\n" % (bench.kernel_source_hash(), label))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "f" * 16)
    assert bench.recorded_traffic(label) is None  # sources changed since the capture
    table.write_text("kernel_source_sha256_16: %s\n%s: 123456\n" % ("f" * 16, label))
    assert bench.recorded_traffic(label) == 123456
    assert bench.recorded_traffic("unknown_label") is None


def test_committed_traffic_table_matches_the_sources():
    """profiles/dram_traffic.txt was captured on the kernel sources as committed."""
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        pytest.skip("no traffic table")
    assert bench.recorded_traffic("mrope_neox_bf16_32768tok_28q4k_h128_s16_24_24") is not None


def test_threaded_oracle_driver_is_bit_exact_with_one_thread():
    """The all-cores CPU baseline cuts a workload into token shards and runs the
    oracle on each in its own thread; the pieces put together are bit-exact with
    one call on the whole workload."""
    from parity import same_bits
    inplace = W.inplace_case("shards_inplace", 31, (2, 37, 3, 64), 16, 48, torch.bfloat16, torch.float32)
    per_head = W.inplace_case("shards_per_head", 32, (2, 9, 3, 32), 0, 0, torch.float16, torch.float16,
                              cs_shape=(2, 9, 3, 32))
    assert same_bits(bench.run_oracle_threaded(inplace, 5), bench.run_oracle(inplace))
    assert same_bits(bench.run_oracle_threaded(per_head, 4), bench.run_oracle(per_head))
    for c in (W.cache_case("shards_neox", 33, 101, 4, 2, 128, 64, 300, torch.bfloat16, True),
              W.cache_case("shards_mrope", 34, 57, 3, 1, 128, 128, 200, torch.float32, True,
                           mrope_section=[16, 24, 24])):
        q1, k1 = bench.run_oracle(c)
        qn, kn = bench.run_oracle_threaded(c, 6)
        assert same_bits(qn, q1) and same_bits(kn, k1)
    assert len(bench.oracle_shards(inplace, 100)) == 37  # never an empty shard


def test_host_cpu_description():
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and 1 <= h["usable_cores"] <= h["nproc"] and h["cpu_model"]


def test_small_call_workloads_and_their_bytes():
    """The small-call table: the [1,16,2,64] f32 workload in its three variants,
    then decode batches of every cache-op head layout and of the fused op."""
    ws = bench.small_workloads()
    names = [w.name for w in ws]
    assert names[:3] == ["inplace_f32_1x16x2x64_slice16_48", "inplace_f32_1x16x2x64_slice0_0",
                         "inplace_f32_1x16x2x64_slice8_8"]
    assert bench.algorithmic_bytes(ws[0]) == 12288 and bench.algorithmic_bytes(ws[1]) == 24576
    assert (ws[2].start, ws[2].end) == (8, 8)
    for T in bench.DECODE_TOKENS:
        neox = ws[names.index("decode_rope_neox_bf16_%dtok_32q8k_h128" % T)]
        assert bench.algorithmic_bytes(neox) == T * (40 * 128 * 2 * 2 + 128 * 2 + 8)
        gptj = ws[names.index("decode_rope_gptj_f16_%dtok_16q16k_h256_r64" % T)]
        assert bench.algorithmic_bytes(gptj) == T * (32 * 64 * 2 * 2 + 64 * 2 + 8)
        mrope = ws[names.index("decode_mrope_neox_bf16_%dtok_28q4k_h128_s16_24_24" % T)]
        assert bench.algorithmic_bytes(mrope) == T * (32 * 128 * 2 * 2 + 128 * 2 + 3 * 8)
        qkv = ws[names.index("decode_qkv_rmsnorm_rope_bf16_%dseq_32q8k8v_h128" % T)]
        assert qkv.tokens == T and int((qkv.slot_mapping >= 0).sum()) == T


def test_source_hash_ignores_comments_and_layout():
    a = "int f(int x) {  // twice x\n  return 2 * x; /* done */ }\n"
    b = "int f(int x) {\n/* a different comment */ return 2 *\n x; }"
    assert bench.source_tokens(a) == bench.source_tokens(b)
    assert bench.source_tokens(a) != bench.source_tokens(a.replace("2 * x", "3 * x"))


def test_the_unhashed_argument_checks_hold_no_kernel_or_launch():
    """The profile hash leaves out the C ABI's argument checks; that file must
    stay host-only code that neither defines nor launches a kernel, nor sizes a
    launch, or a change there could alter what the profiles measured."""
    path = os.path.join(os.path.dirname(bench.__file__), "transformer_rope_positional_gb300", "csrc",
                        bench.ARGUMENT_CHECKS)
    code = bench.source_tokens(open(path).read())
    for marker in ("__global__", "__device__", "<<<", "cudaLaunch", "resident_blocks", "sm_count", "opt_in_shared",
                   "cudaFuncSetAttribute", "__launch_bounds__"):
        assert marker not in code, marker
    csrc = os.path.dirname(path)
    hashed = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")) and n != bench.ARGUMENT_CHECKS]
    assert {"rope_cache.cu", "rope_qkv.cu", "rope_launch.cu", "rope_inplace.cuh", "rope_device.cuh"} <= set(hashed)


def test_reference_arm_reports_the_same_config_as_ours():
    """The reference arm (the oracle on the host cores) prints the config that
    our arm prints: the same workload, bytes and tokens per step."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(bench.__file__)
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--reference-seconds", "0.5"], capture_output=True, text=True, check=True,
                         cwd=root, timeout=600).stdout
    line = json.loads(out.strip().splitlines()[-1])
    cases = bench.build_workloads()
    assert line["impl"] == "reference"
    assert line["config"] == bench.step_config(sum(bench.algorithmic_bytes(c) for c in cases),
                                               sum(c.tokens for c in cases))
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_library_builds_of_concurrent_processes_take_turns(tmp_path, monkeypatch):
    """Ranks of a multi-GPU run build at once; the shared object files must not
    be compiled by two of them together (the build holds a lock file)."""
    import threading
    import time

    from transformer_rope_positional_gb300 import build as B

    monkeypatch.setattr(B, "LIB_DIR", str(tmp_path))
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "librope_gb300.so"))
    inside, most, calls = [0], [0], []
    guard = threading.Lock()

    def fake_build(lib_path, verbose, debug):
        with guard:
            inside[0] += 1
            most[0] = max(most[0], inside[0])
        time.sleep(0.2)
        with guard:
            inside[0] -= 1
            calls.append(lib_path)
        return lib_path

    monkeypatch.setattr(B, "_build_locked", fake_build)
    threads = [threading.Thread(target=B.build, kwargs={"force": True}) for _ in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert len(calls) == 4 and most[0] == 1
