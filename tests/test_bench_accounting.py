"""The benchmark's algorithmic work per step (the numerator of every roofline figure it prints),
checked on the CPU against counts worked out by hand from the workload shapes:

  decode CSA at 128K, batch 16 (E = 32768 entries, top-k 512, window 128, d = 128, 64 heads,
  indexer 4 heads x 64 FP4):
    index keys  32768 x (32 B codes + 2 B scales)                 = 1,114,112 B per sequence
    queries     4 heads x 34 B                                    =       136 B
    scores      32768 x 2 B written (read back by the top-k)      =    65,536 B
    top-k       32768 x 2 B read + 512 x 4 B written              =    67,584 B
    attention   (512 + 128) keys x (K + V rows of 256 B)          =   327,680 B, + Q/O 32,768 B
  decode HCA at 1M, batch 32 (8192 entries + 128 window keys)     = 4,292,608 B per sequence
  prefill chunk of 8192 queries at 128K: indexer sum_t 2 * 4 * 64 * floor((t+1)/4) over
  t = 122880 .. 131071, attention 8192 x 64 heads x (2048 + 128) keys x 128 x 4 FLOPs."""
import bench
from synth import get_config


def test_csa_decode_128k_work():
    w = bench.step_work(get_config("csa_decode_128k"))
    B = 16
    assert w["indexer_mxf4"]["bytes"] == B * (1_114_112 + 136 + 65_536)
    assert w["indexer_mxf4"]["flops"] == B * 2 * 4 * 64 * 32768
    assert w["topk"]["bytes"] == B * 67_584
    assert w["csa_attend"]["bytes"] == B * (327_680 + 32_768)
    assert w["csa_attend"]["flops"] == B * 4 * 64 * 128 * 640
    # one block of 4 tokens pooled per sequence: 4 x (K + V rows + logit) read, one entry written
    assert w["compress"]["bytes"] == B * (4 * (512 + 4) + 512)
    assert bench.units_per_step(get_config("csa_decode_128k")) == (16, "tok/s")


def test_hca_decode_1m_work():
    w = bench.step_work(get_config("hca_decode_1m"))
    assert w["hca_attend"]["bytes"] == 32 * 4_292_608
    assert w["hca_attend"]["flops"] == 32 * 4 * 64 * 128 * (8192 + 128)


def test_prefill_flops():
    w = bench.step_work(get_config("csa_prefill_8k_of_128k"))
    vis = sum((t + 1) // 4 for t in range(122880, 131072))
    assert w["indexer_mxf4"]["flops"] == 2 * 4 * 64 * vis          # 133.1 GFLOP
    assert w["csa_attend"]["flops"] == 8192 * 64 * 2176 * 128 * 4   # 584.1 GFLOP
    assert bench.units_per_step(get_config("csa_prefill_8k_of_128k")) == (None, "TFLOP/s")


def test_optional_rows_add_their_kernels():
    s = get_config("csa_prefill_8k_of_128k").layer("csa")
    w = bench.layer_work(s, index_keys=True)
    # the chunk's 2048 blocks: 4 index-key rows of 128 B + 4 logits read, 34 B of keys written
    assert w["index_keys"]["bytes"] == 2048 * (4 * (128 + 4) + 34)
    assert "index_keys" not in bench.layer_work(s)


def test_fused_decode_kernel_work_is_its_steps_without_the_score_round_trip():
    # one launch scores, selects and attends: its bytes are the three steps' bytes less the
    # BF16 scores the separate kernels write and read back (32768 x 2 B x 2 per sequence)
    wl = get_config("csa_decode_128k")
    w = bench.kernel_work(wl, bench.step_work(wl))
    B = 16
    parts = w["indexer_mxf4"]["bytes"] + w["topk"]["bytes"] + w["csa_attend"]["bytes"]
    assert w["csa_decode"]["bytes"] == parts - B * 32768 * 4
    assert w["csa_decode"]["flops"] == w["indexer_mxf4"]["flops"] + w["csa_attend"]["flops"]
    assert w["indexer_topk"]["bytes"] == w["indexer_mxf4"]["bytes"] + w["topk"]["bytes"]


def test_step_totals_count_each_step_once():
    wl = get_config("csa_prefill_8k_of_128k")
    w = bench.step_work(wl)
    assert "csa_decode" not in w and "indexer_topk" not in w
    assert sum(v["flops"] for v in w.values()) == w["indexer_mxf4"]["flops"] + \
        w["csa_attend"]["flops"] + w["compress"]["flops"]
