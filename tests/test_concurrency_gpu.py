"""Concurrent calls: host threads, each on its own CUDA stream.

The library keeps no per-call state outside the caller's buffers (the tensor
map and planner caches are locked, one-time kernel setup runs once), so
calls from several host threads on several streams at the same time must
give exactly what the same calls give one after another.  A worker's first
CUDA work may be a library call, with no context current in that thread yet:
the driver's tensor-map encoding then has to make the primary context current
itself.  Each thread runs its job (fp32 decode, bf16 decode in its
one-long-request shape, 4-bit decode, prefill at D = 64 and 128, the
quantizer) several times into its own output and workspace; the outputs must
equal the sequential ones bit for bit.  The plan overrides are process-wide
settings and are not used here.
"""

import threading

import pytest
import torch

from gqa_attention_kv_decode_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
REPEATS = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def make_jobs():
    jobs = []

    def decode_job(dtype, B, S, layer):
        q, k, v = inputs.qkv(B, 28, 4, 128, 1, S, dtype, layer=layer, device=DEV)
        ws = binding.decode_workspace(B, 28, 4, 128, S, binding._dtype_code(q), DEV)

        def run(o, stream):
            ws.zero_()  # (the status word must start at zero; the rest is scratch)
            binding.gqa_attn_decode(q, k, v, o, None, 128 ** -0.5, ws, stream=stream)
        return run, torch.empty_like(q)

    jobs.append(decode_job(torch.float32, 2, 4096, 121))
    jobs.append(decode_job(torch.bfloat16, 1, 16384, 122))

    kc, ks, kb, vc, vs, vb = inputs.q4_cache(2, 8, 128, 2048, layer=123, device=DEV)
    q4 = inputs.randn((2, 32, 1, 128), 124, torch.bfloat16, DEV)
    ws4 = binding.decode_q4_workspace(2, 32, 8, 128, 2048, DEV)

    def q4_run(o, stream):
        ws4.zero_()
        binding.gqa_attn_decode_q4(q4, kc, ks, kb, vc, vs, vb, o, None, 128 ** -0.5, ws4, stream=stream)
    jobs.append((q4_run, torch.empty_like(q4)))

    for D, T, seed in ((64, 1024, 125), (128, 600, 126)):
        qp = inputs.randn((1, 14, T, D), seed, torch.bfloat16, DEV)
        kp = inputs.randn((1, 2, T, D), seed + 10, torch.bfloat16, DEV)
        vp = inputs.randn((1, 2, T, D), seed + 20, torch.bfloat16, DEV)

        def pf_run(o, stream, qp=qp, kp=kp, vp=vp, T=T, D=D):
            binding.gqa_attn_prefill(qp, kp, vp, o, T, D ** -0.5, True, stream=stream)
        jobs.append((pf_run, torch.empty_like(qp)))

    src = inputs.randn((2, 8, 1024, 128), 127, torch.bfloat16, DEV)
    codes = torch.empty((2, 8, 1024, 64), dtype=torch.uint8, device=DEV)
    scale = torch.empty((2, 8, 1024, 2), dtype=torch.float16, device=DEV)
    bias = torch.empty_like(scale)

    def quant_run(o, stream):
        binding.gqa_attn_quantize_q4(src, codes, scale, bias, stream=stream)
        o.copy_(codes)
    jobs.append((quant_run, torch.empty_like(codes)))
    return jobs


def test_concurrent_calls_equal_sequential_calls():
    jobs = make_jobs()
    torch.cuda.synchronize()
    # one after another, on the default stream
    refs = []
    for run, out in jobs:
        run(out, torch.cuda.current_stream())
        torch.cuda.synchronize()
        refs.append(out.clone())
    # all at once: one host thread and one stream per job, released together
    outs = [torch.full_like(out, 0) for _, out in jobs]
    start = threading.Barrier(len(jobs))
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream(DEV)
            run, _ = jobs[i]
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(REPEATS):
                    run(outs[i], stream)
            stream.synchronize()
        except Exception as e:  # reported below, with the job's index
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    torch.cuda.synchronize()
    assert not errors, errors
    for i, (got, ref) in enumerate(zip(outs, refs)):
        assert torch.equal(got, ref), f"job {i} differs when run concurrently"
