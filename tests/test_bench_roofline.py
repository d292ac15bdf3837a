"""The bench's roofline arithmetic on the CPU, against figures worked out by hand."""
import pytest

import bench

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


@pytest.mark.parametrize("V,chunks", [(2048, 8), (32768, 64), (262144, 74), (1000, 4), (100, 1)])
def test_vocab_chunks_match_the_library_layout(V, chunks):
    # 256-column tiles split into at most 76 chunks of equal tile counts:
    # 2048 -> 8 tiles, 1 each; 32768 -> 128 tiles, 2 each; 262144 -> 1024 tiles, 14 each -> 74 chunks
    assert bench.vocab_chunks(V) == chunks


def test_one_canvas_at_v32k_is_bound_by_the_w_stream():
    # W 32768 x 1024 bf16 = 64 MiB; fp32 residual 256 x 1024 x 4 = 1 MiB; norm weights 4 KiB;
    # partial records 256 x 64 x 32 B = 512 KiB
    roof, t_hbm, t_tc = bench.lmhead_roofline(32768, 1024, 256, True, 40e-6, PEAKS)
    want_bytes = 64 * 2**20 + 2**20 + 4096 + 512 * 1024
    assert roof["algorithmic_bytes_per_launch"] == want_bytes
    assert roof["algorithmic_flops_per_launch"] == 2.0 * 256 * 32768 * 1024
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s" and t_hbm > t_tc
    assert roof["achieved"] == pytest.approx(want_bytes / 40e-6 / 1e9)
    assert roof["frac"] == pytest.approx(want_bytes / 40e-6 / 6800e9)


def test_sixteen_canvases_at_model_scale_are_bound_by_the_tensor_pipe():
    # 4096 positions reuse each W row 4096 times: 2 x 4096 x 262144 x 2816 flops at 1900 TFLOP/s
    # take 3.18 ms, the 1.5 GB of W at 6800 GB/s 0.23 ms
    flops = 2.0 * 4096 * 262144 * 2816
    roof, t_hbm, t_tc = bench.lmhead_roofline(262144, 2816, 4096, True, 3.9e-3, PEAKS)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert t_tc == pytest.approx(flops / 1900e12) and t_hbm < t_tc
    assert roof["frac"] == pytest.approx(flops / 3.9e-3 / 1900e12)


def test_single_cta_kernel_reads_bf16_rows_instead_of_the_residual():
    # below 256 positions the RMSNorm kernel writes h first: the LM head reads 16 x 128 bf16 rows
    roof, _, _ = bench.lmhead_roofline(2048, 128, 16, False, 5e-6, PEAKS)
    assert roof["algorithmic_bytes_per_launch"] == 2048 * 128 * 2 + 16 * 128 * 2 + 16 * 8 * 32


def test_self_conditioning_roofline_counts_both_contractions():
    # one canvas at model scale: W 262144 x 2816 bf16 once, the bf16 rows h (256 x 2816 x 2 B) and
    # the fp32 output (256 x 2816 x 4 B); the logits and P W are 2 x 2 x 256 x 262144 x 2816 flops,
    # 0.398 ms at 1900 TFLOP/s against 0.218 ms for the bytes at 6800 GB/s: tensor-bound
    V, d, P = 262144, 2816, 256
    r = bench.self_cond_roofline(V, d, P, 0.56e-3, PEAKS)
    want_bytes = V * d * 2 + P * d * 2 + P * d * 4
    flops = 4.0 * P * V * d
    assert r["algorithmic_bytes_per_call"] == want_bytes and r["algorithmic_flops_per_call"] == flops
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["roofline_time_ms"] == pytest.approx(flops / 1900e12 * 1e3)
    assert r["frac"] == pytest.approx(flops / 0.56e-3 / 1900e12)


def test_self_conditioning_roofline_at_few_positions_is_bound_by_w():
    # 16 positions: the flops (2 x 2 x 16 x 2048 x 128) take nanoseconds, W 2048 x 128 bf16 microseconds
    r = bench.self_cond_roofline(2048, 128, 16, 10e-6, PEAKS)
    want_bytes = 2048 * 128 * 2 + 16 * 128 * 6
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(want_bytes / 10e-6 / 1e9)


def test_topk_self_conditioning_roofline():
    # one canvas at model scale: 2 x 256 x 262144 x 2816 = 378 GFLOP take 0.2 ms at 1900 TF/s, while W
    # (1.476 GB) plus the 32 gathered rows per position take 0.22 ms at 6800 GB/s: bound by W
    r = bench.self_cond_topk_roofline(262144, 2816, 256, 32, 0.5e-3, PEAKS)
    want = 262144 * 2816 * 2 + 256 * 2816 * 6 + 256 * 32 * 2816 * 2
    assert r["bound"] == "hbm" and r["algorithmic_bytes_per_call"] == want
    assert r["frac"] == pytest.approx(want / 0.5e-3 / 6800e9)
    # K above V keeps V rows
    assert bench.self_cond_topk_roofline(200, 64, 16, 256, 1e-5, PEAKS)["algorithmic_bytes_per_call"] == \
        200 * 64 * 2 + 16 * 64 * 6 + 16 * 200 * 64 * 2
    # sixteen canvases: 6.05 PFLOP take 3.2 ms, 2.28 GB 0.34 ms: the contraction bounds it
    r = bench.self_cond_topk_roofline(262144, 2816, 4096, 32, 4e-3, PEAKS)
    assert r["bound"] == "tensor" and r["achieved"] == pytest.approx(2 * 4096 * 262144 * 2816 / 4e-3 / 1e12)


def test_kernel_digest_ignores_comments_but_not_code():
    src = 'int a = 1;  // a note\n/* a block\n   note */\nconst char* s = "x // y /* z */";\n\n  b += 2;\n'
    assert bench.strip_comments(src) == 'int a = 1;\nconst char* s = "x // y /* z */";\n  b += 2;'
    assert bench.strip_comments(src.replace("a note", "another note")) == bench.strip_comments(src)
    assert bench.strip_comments(src.replace("b += 2", "b += 3")) != bench.strip_comments(src)
