"""Host-side arithmetic of the benchmark, pinned to hand-computed closed forms:
the algorithmic bytes behind the roofline fraction, the RDKV flop count, the
ncu traffic records and the workload keys both benchmark arms print."""
import argparse

import numpy as np
import pytest

import bench
from quantized_kv_cache_11_gb300 import synthetic as S


def test_decode_bytes_128k_2bit_by_hand():
    # 131,008 quantized tokens + 64 fp16 tail tokens, 8 KV heads, D 128, 2 bits
    codes = 2 * 131008 * 8 * 128 * 2 // 8          # K and V codes
    k_meta = (131008 // 32) * 8 * 128 * 2 * 2      # fp16 scale + zero per channel per key group
    v_meta = 131008 * 8 * (128 // 32) * 2 * 2      # fp16 scale + zero per 32 channels per token
    tail = 64 * 8 * 128 * 2 * 2                    # fp16 K and V rows
    q_out = 32 * 128 * (2 + 4)                     # fp16 q in, fp32 out
    assert codes + k_meta + v_meta + tail + q_out == 100_900_864
    assert bench.algorithmic_bytes(S.LLAMA31_8B_128K, 131008, 64) == 100_900_864


def test_decode_bytes_128k_4bit_and_mha_by_hand():
    codes4 = 2 * 131008 * 8 * 128 * 4 // 8
    meta = 2 * 16_769_024
    assert bench.algorithmic_bytes(S.LLAMA31_8B_128K_4BIT, 131008, 64) == codes4 + meta + 262_144 + 24_576
    # 8 sequences x 40 heads (MHA), 4,064 quantized + 32 tail tokens, 2 bits
    w = S.LLAMA2_13B
    per_head = 2 * 4064 * 128 * 2 // 8 + (4064 // 32) * 128 * 4 + 4064 * 4 * 4 + 32 * 128 * 4
    assert bench.algorithmic_bytes(w, 4064, 32) == 8 * 40 * per_head + 8 * 40 * 128 * 6


def test_decode_bytes_with_sink_window():
    # sink tokens are fp16 rows like the tail
    base = bench.algorithmic_bytes(S.LLAMA31_8B_128K, 131008, 60)
    assert bench.algorithmic_bytes(S.LLAMA31_8B_128K, 131008, 60, 4) == base + 4 * 8 * 128 * 4


def test_prefill_bytes_of_the_serving_chunks_by_hand():
    # 16 full 32,768-token chunks at 4 bits: fp16 K and V in, codes + metadata out
    w = S.SERVING
    read = 2 * 16 * 32768 * 8 * 128 * 2
    write = 2 * 16 * 32768 * 8 * 128 * 4 // 8 + 16 * 1024 * 8 * 128 * 4 + 16 * 32768 * 8 * 4 * 4
    assert (read, write) == (2_147_483_648, 671_088_640)
    assert bench.prefill_algorithmic_bytes(w.scaled(batch=16), 32768, 0) == read + write


def test_rdkv_flops_by_hand():
    # 4 x 32 query heads, 65,536 positions: causal pairs T(T+1)/2, 2D flops each
    assert bench.rdkv_flops(S.TRIZONE) == 4 * 32 * (65536 * 65537 // 2) * 2 * 128


def test_traffic_record_requires_the_measured_source():
    sha = bench._kernel_sha()
    name = f"decode_traffic_{S.LLAMA31_8B_128K.name}.txt"
    rec = bench.read_traffic(name, S.LLAMA31_8B_128K.name, sha)
    assert rec is None or rec > bench.algorithmic_bytes(S.LLAMA31_8B_128K, 131008, 64)
    assert bench.read_traffic(name, S.LLAMA31_8B_128K.name, "0" * 16) is None
    assert bench.read_traffic(name, "another_workload", sha) is None
    assert bench.read_traffic("no_such_record.txt", S.LLAMA31_8B_128K.name, sha) is None


@pytest.mark.parametrize("rope,sink", [(0.0, 0), (500000.0, 0), (0.0, 4)])
def test_both_arms_name_the_workload_alike(rope, sink):
    # the reference arm builds its config with the same helper as the GPU arm
    args = argparse.Namespace(rope=rope, sink=sink, bits=2)
    w = bench.workload(2)
    cfg = bench.uniform_config(w, args, 131008, 64 - sink, sink)
    assert cfg["workload"].endswith("_prerope") == bool(rope)
    assert cfg["n_quant"] + cfg["n_tail"] + cfg["n_sink"] == w.context
    assert {"l2", "launch"}.isdisjoint(cfg)


def test_sink_window_keeps_the_quantized_region():
    # a 4-token window at the front takes its tokens out of the tail: the
    # 131,008 quantized tokens stay, the tail drops from 64 to 60
    inp = {"seq_len": np.array([131072, 1000], np.int32), "n_tail": np.array([64, 8], np.int32)}
    out = bench.with_sink(inp, 4)
    assert out["n_tail"].tolist() == [60, 4]
    assert (out["seq_len"] - out["n_tail"] - 4).tolist() == [131008, 992]
    # no tail to give: the window cannot be carved out without shrinking the groups
    with pytest.raises(ValueError):
        bench.with_sink({"seq_len": np.array([256], np.int32), "n_tail": np.array([0], np.int32)}, 5)


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = tmp_path / "quantized_kv_cache_11_gb300" / "csrc"
    src.mkdir(parents=True)
    body = "// header comment\nint f(int x) {  /* block\n   comment */ return x + 1; }\n"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (src / "k.cu").write_text(body)
    h0 = bench._kernel_sha(("k.cu",))
    (src / "k.cu").write_text(body.replace("header comment", "another note").replace("  /*", "\n\n  /*"))
    assert bench._kernel_sha(("k.cu",)) == h0      # comments and blank lines only
    (src / "k.cu").write_text(body.replace("x + 1", "x + 2"))
    assert bench._kernel_sha(("k.cu",)) != h0      # the code itself
