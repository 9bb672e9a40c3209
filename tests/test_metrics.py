"""Byte and flop accounting pinned to figures the pages print."""

from gqa_attention_kv_decode_gb300 import metrics


def test_kv_bytes_match_decode_page():
    # "2x Faster Qwen2 Decode on Metal in Candle", "Why It Matters":
    # 2 (K, V) x 4 KV heads x 2048 tokens x 128 dim x 4 bytes = 8 MiB / layer
    assert metrics.decode_kv_bytes(4, 128, 2048, 4) == 8 * 2**20
    # and the 7x expanded copy: 56 MiB / layer, 1.53 GiB over 28 layers
    expanded = 7 * metrics.decode_kv_bytes(4, 128, 2048, 4)
    assert expanded == 56 * 2**20
    assert abs(28 * expanded / 2**30 - 1.53) < 0.01


def test_score_matrix_bytes_match_prefill_page():
    # "Fused attention makes a 4,096-token Qwen2 prefill ...", "Why it matters":
    # a [14, T, T] score matrix is 470 MB at T = 4,096 (bf16)
    b = metrics.score_matrix_bytes(14, 4096, 4096, 2)
    assert round(b / 1e6) == 470


def test_decode_bytes_include_q_and_o():
    assert metrics.decode_bytes(28, 4, 128, [2048], 4) == 8 * 2**20 + 2 * 28 * 128 * 4


def test_visible_pairs_closed_form():
    # brute force count of j <= i + off
    for q_len, kv_len in [(1, 7), (5, 5), (3, 10), (513, 513)]:
        off = kv_len - q_len
        brute = sum(1 for i in range(q_len) for j in range(kv_len) if j <= i + off)
        assert metrics.prefill_visible_pairs(q_len, kv_len) == brute
    assert metrics.prefill_visible_pairs(4, 9, causal=False) == 36


def test_chunk_flops():
    # 512-query chunk at offset 3584 of 4096 keys: 1,966,336 visible pairs
    assert metrics.prefill_visible_pairs(512, 4096) == 1966336
    assert abs(metrics.prefill_flops(14, 64, 512, 4096) / 1e9 - 7.05) < 0.01


def test_q4_row_bytes():
    # 64 bytes of codes + 2 groups x (fp16 scale + fp16 bias) = 72 B per row
    assert metrics.q4_row_bytes(128, 64) == 72


def test_quantize_bytes_per_row():
    # a D=128 bf16 row is read (256 B) and written as 64 code bytes plus two
    # fp16 (scale, bias) pairs: 256 + 64 + 8
    assert metrics.quantize_bytes(1, 128) == 328
    assert metrics.quantize_bytes(10, 64) == 10 * (128 + 32 + 4)


def test_bench_kernel_cases_do_not_shadow_the_workload_constants():
    """`bench.py --kernel CASE` builds its inputs in one function; a local
    name equal to a module constant (D, HQ, ...) makes that constant local to
    the whole function and breaks the other cases at run time."""
    import symtable

    import bench

    src = open(bench.__file__).read()
    top = symtable.symtable(src, bench.__file__, "exec")
    fn = next(c for c in top.get_children() if c.get_name() == "_case_inputs")
    constants = {"D", "HQ", "HKV", "S_HEAD", "LAYERS", "PREFILL_LAYERS"}
    assert not (constants & set(fn.get_locals())), constants & set(fn.get_locals())
    for case in bench.KERNEL_CASES:
        assert case.split("-")[0] in {"decode", "q4", "quantize", "prefill", "varlen"}
