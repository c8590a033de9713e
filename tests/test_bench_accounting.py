"""Host logic of bench.py (CPU): the algorithmic work it divides by, checked against the
figures worked out from the block's shapes (41,943,040 parameters, causal pairs T(T+1)/2 per
head, bf16 K/V cache of 8 heads x 128), and the sizing of the oracle's timed prefix."""
import pytest

import bench
from transformer_gqa_attention_gb300 import inputs as gin


def test_prefill_flops_of_the_workloads():
    # projections 2 x 41,943,040 per token; causal attention 4 x 128 x 32 x T(T+1)/2 per sequence
    # = 8192 T(T+1); the rounded totals are the ones worked out for the workloads (GFLOP)
    for (B, T, proj_g, attn_g) in [(1, 16, 1.342, 0.002228), (1, 2048, 171.80, 34.38),
                                   (4, 8192, 2748.78, 2199.29), (1, 32768, 2748.78, 8796.36)]:
        proj, attn = bench.prefill_flops(B, T)
        assert proj == 2 * 41_943_040 * B * T
        assert attn == 8192 * T * (T + 1) * B
        assert abs(proj / 1e9 - proj_g) < 0.01 * proj_g and abs(attn / 1e9 - attn_g) < 0.001 * attn_g
    # a causal prefix continuing a cache sees its start_pos earlier keys in full
    _, a = bench.prefill_flops(1, 1, start_pos=9)
    assert a == 4 * 128 * 32 * 10
    _, a_nc = bench.prefill_flops(1, 4, causal=False)
    assert a_nc == 4 * 128 * 32 * 16


def test_decode_bytes_of_the_workload():
    # KV 64 x 4096 x 8 x 128 x 2 B x 2 + weights 2 x 41,943,040 B + x in + Delta out + new K/V
    assert bench.decode_bytes(64, 4096) == 1_159_462_912


def test_kernel_work_models():
    w = gin.WORKLOADS["prefill_b1_t2048"]
    assert bench.kernel_work("qkv_gemm", w) == ("tensor", 2.0 * 2048 * 4096 * 6144, "TFLOP/s")
    assert bench.kernel_work("out_gemm", w)[1] == 2.0 * 2048 * 4096 * 4096
    assert bench.kernel_work("flash_prefill", w)[1] == 8192 * 2048 * 2049
    d = gin.WORKLOADS["decode_b64_pos4095"]
    # K and V of 4096 positions, q read and H written (64 x 4096 bf16 each)
    assert bench.kernel_work("decode_attn", d) == ("hbm", float(64 * 4096 * 8 * 128 * 4 + 2 * 64 * 4096 * 2), "GB/s")
    # a 16-token prefill runs the same kernel: the 16 cached positions, 16 query rows in and out
    s = gin.WORKLOADS["prefill_b1_t16"]
    assert bench.kernel_work("decode_attn", s)[1] == float(16 * 8 * 128 * 4 + 2 * 16 * 4096 * 2)
    assert bench.kernel_work("nonexistent", d) == (None, None, None)


def test_prefix_sizing_follows_the_quadratic_model():
    # times generated from t(n) = a n + b n^2: the chosen prefix meets the budget
    a, b = 1e-3, 2e-6
    t = lambda n: a * n + b * n * n
    n = bench.prefix_for_budget(512, t(512), 1024, t(1024), 5.0, 32768)
    assert t(n) <= 5.0 < t(n + 2)
    # a linear model would have picked ~5000 positions here; the cap and T bound it
    assert bench.prefix_for_budget(512, t(512), 1024, t(1024), 1e6, 32768) == 4096
    assert bench.prefix_for_budget(512, t(512), 1024, t(1024), 1e6, 700) == 700
    assert bench.prefix_for_budget(512, t(512), 1024, t(1024), 1e-9, 32768) == 16


@pytest.mark.parametrize("name", sorted(gin.WORKLOADS))
def test_workload_config_names_the_workload(name):
    w = gin.WORKLOADS[name]
    c = bench.workload_config(w)
    assert c["workload"] == name and c["B"] == w.B and c["T"] == w.T and c["S_max"] == w.s_max


def test_shard_accounting_is_the_whole_divided_by_the_split():
    for n in (1, 2, 4):
        p8, a8 = bench.prefill_flops(1, 2048)
        pn, an = bench.prefill_flops(1, 2048, n_kv=n)
        assert pn * 8 == p8 * n and an * 8 == a8 * n
    # a decode shard reads its share of the cache and of the weights; x and Delta stay whole
    whole = bench.decode_bytes(64, 4096)
    part = bench.decode_bytes(64, 4096, n_kv=1)
    assert part == 64 * 4096 * 128 * 4 + 41_943_040 * 2 // 8 + 64 * 4096 * 6 + 64 * 128 * 4
    assert part < whole / 7
    w = gin.WORKLOADS["prefill_b1_t2048_tp8"]
    assert bench.kernel_work("qkv_gemm", w)[1] == 2.0 * 2048 * 4096 * 768
    assert bench.kernel_work("out_gemm", w)[1] == 2.0 * 2048 * 512 * 4096


def test_chunked_prefill_workloads_accounting():
    # the last 2048-token chunk of a 32768-token prompt: each row t sees 30720 + t + 1 keys
    w = gin.WORKLOADS["prefill_b1_t2048_pos30720"]
    proj, attn = bench.prefill_flops(w.B, w.T, w.start_pos, w.causal)
    assert proj == 2 * 41_943_040 * 2048
    assert attn == 4 * 128 * 32 * sum(30720 + t + 1 for t in range(2048))
    # 16 tokens after 4080 cached positions run the four-position kernel: K and V of all 4096
    # positions of the 4 sequences once, q in and H out
    s = gin.WORKLOADS["prefill_b4_t16_pos4080"]
    assert bench.kernel_work("decode_attn", s)[1] == float(4 * 4096 * 8 * 128 * 4 + 2 * 64 * 4096 * 2)
    inp = gin.make_inputs(s)
    assert inp.cache_k.shape == (4, 4096, 8, 128) and inp.R.shape == (16, 64, 2)


def test_source_digest_ignores_comments_only():
    code = 'int f(int a) {  // add one\n  return a + 1;  /* done */\n}\nconst char* s = "// kept";\n'
    assert bench._code_only(code) == bench._code_only(code.replace("add one", "increment").replace("done", "ok") + "\n\n")
    assert bench._code_only(code) != bench._code_only(code.replace("a + 1", "a + 2"))
    assert '"// kept"' in bench._code_only(code)
