"""The benchmark's algorithmic bytes and FLOPs against closed forms.

Every roofline fraction bench.py reports divides these counts by a measured
time, so they are pinned here to the layer's arithmetic written out by hand:
per expert 2I x H codes for gate/up and H x I for down at half a byte each,
one bf16 scale per 128 codes; 2 FLOPs per multiply-add.
"""
import numpy as np

import bench
import moe_synth as ms

MEASURED = {"hbm_gbs": 6795.5, "bf16_tflops": 1885.7, "source": "measured"}


def test_expert_bytes_of_the_v4_flash_shape():
    shape = ms.CONFIGS["decode1"]
    w13, w2 = bench.expert_bytes(shape, shape.inter)
    assert w13 == 2 * 2048 * 4096 // 2 + 2 * 2048 * 32 * 2 == 8_650_752
    assert w2 == 4096 * 2048 // 2 + 4096 * 16 * 2 == 4_325_376
    assert w13 + w2 == 12_976_128


def _counts(shape, hit):
    c = np.zeros(shape.experts, np.int64)
    c[:hit] = 1
    return c


def test_decode1_layer_work():
    shape = ms.CONFIGS["decode1"]
    work = bench.layer_work(shape, _counts(shape, 6))
    # six routed experts plus the shared one, the fp32 router and its bias,
    # one bf16 token in and out
    assert work["hit"] == 6
    assert work["bytes"] == 7 * 12_976_128 + (256 * 4096 * 4 + 256 * 4) + 2 * 4096 * 2
    assert work["bytes"] == 95_044_608
    # router 2·T·E·H plus 2·3·H·I per (token, expert), shared included
    assert work["flops"] == 2 * 256 * 4096 + 7 * 2 * 3 * 4096 * 2048 == 354_418_688


def test_prefill8192_flops_are_2_903_tflop():
    shape = ms.CONFIGS["prefill8192"]
    work = bench.layer_work(shape, np.full(shape.experts, 8192 * 6 // 256))
    assert work["hit"] == 256
    assert work["flops"] == 2 * 8192 * 256 * 4096 + 8192 * 7 * 50_331_648
    assert abs(work["flops"] / 1e12 - 2.903) < 1e-3


def test_expert_kernel_flops_split_two_thirds_one_third():
    shape = ms.CONFIGS["prefill8192"]
    work = bench.layer_work(shape, np.full(shape.experts, 192))
    _, f13 = bench.kernel_work("tc_gate_up_swiglu", shape, work)
    _, f2 = bench.kernel_work("tc_down", shape, work)
    _, fr = bench.kernel_work("router_logits_tc", shape, work)
    assert f13 == 2 * f2
    assert f13 + f2 + fr == work["flops"]


def test_decode_kernel_counts_the_whole_layer():
    shape = ms.CONFIGS["decode1"]
    work = bench.layer_work(shape, _counts(shape, 6))
    assert bench.kernel_work("decode_fused", shape, work) == (work["bytes"], work["flops"])


def test_roofline_takes_the_slower_bound():
    d1 = ms.CONFIGS["decode1"]
    w1 = bench.layer_work(d1, _counts(d1, 6))
    r = bench.roofline("decode_fused", d1, w1, 48.4e-6, MEASURED)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 95_044_608 / 48.4e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["achieved"] / 6795.5) < 1e-12
    p = ms.CONFIGS["prefill8192"]
    wp = bench.layer_work(p, np.full(p.experts, 192))
    r = bench.roofline("tc_gate_up_swiglu", p, wp, 1.38e-3, MEASURED)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["frac"] - r["achieved"] / 1885.7) < 1e-12


def test_tensor_core_gate_up_counts_activations_once():
    # the layer reads each token row once; the gathered copy the GEMM reads
    # (T*k + T rows) is reported apart, not as algorithmic bytes
    shape = ms.CONFIGS["prefill8192"]
    work = bench.layer_work(shape, np.full(shape.experts, 192))
    nbytes, _ = bench.kernel_work("tc_gate_up_swiglu", shape, work)
    hrows = 8192 * 6 * 2048 + 8192 * 2048
    assert nbytes == work["w13_bytes"] + 8192 * 4096 * 2 + hrows * 2
    assert bench.implementation_bytes("tc_gate_up_swiglu", shape) == 8192 * 6 * 4096 * 2
    assert bench.implementation_bytes("decode_fused", shape) == 0


def test_both_arms_print_the_same_config():
    import argparse
    args = argparse.Namespace(expert_path="auto")
    shape = ms.CONFIGS["decode1"]
    c = bench.config_of(shape, args)
    assert c["workload"] == "decode1" and c["tokens"] == 1 and c["experts"] == 256


def test_w4a8_kernel_work():
    """The W4A8 path's kernels: the same weight bytes, e4m3 activations (one
    byte, one fp32 scale per 128), fp32 h and y; the fp8 tensor peak is the
    measured bf16 one times the nominal ratio 2."""
    shape = ms.CONFIGS["decode64"]
    work = bench.layer_work(shape, _counts(shape, 150))
    T, H, k, I, Is = 64, 4096, 6, 2048, 2048
    hrows = T * k * I + T * Is
    rows = T * k + T
    b13, f13 = bench.kernel_work("w4a8_gate_up_swiglu", shape, work)
    assert b13 == work["w13_bytes"] + T * H + T * (H // 128) * 4 + hrows * 4
    assert f13 == 2 * H * 2 * hrows
    b2, f2 = bench.kernel_work("w4a8_down", shape, work)
    assert b2 == work["w2_bytes"] + hrows + hrows // 128 * 4 + rows * H * 4
    assert f2 == 2 * H * hrows
    assert bench.kernel_work("w4a8_quantize_x", shape, work) == (T * H * 3 + T * 32 * 4, 0)
    p = ms.CONFIGS["prefill8192"]
    wp = bench.layer_work(p, np.full(p.experts, 192))
    r = bench.roofline("w4a8_gate_up_swiglu", p, wp, 1.0e-3, MEASURED)
    assert r["bound"] == "tensor" and r["peak"] == 2 * 1885.7
