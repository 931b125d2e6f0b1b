"""Calls from several host threads at once, each thread on its own CUDA
stream (the pages' thread-safety fixes: talk slide 10 "70 Fixes to the ROCm
Fork", eight-thread tests that used to fail).  The entry points whose
kernels pass partial sums through global memory -- mx_qmv with K split
across CTAs, mx_moe_down_combine and the NVFP4 mx_quantize -- use a
workspace slot of the stream they are issued on, so every concurrent call
must return exactly the bits a lone call returns."""
import threading

import numpy as np
import pytest

from gemm_decode_register_gb300 import synth
from gpu_util import check_close, dev_bf16, dev_i32, dev_u8, need_gpu

pytestmark = pytest.mark.gpu

THREADS, ITERS = 8, 20


def test_threads_on_their_own_streams(orc):
    torch = need_gpu()
    from gemm_decode_register_gb300 import ops

    F4, NV = synth.FMT_MXFP4, synth.FMT_NVFP4
    # qmv: 4 tokens x K = 28672 cannot be staged in one CTA's shared memory
    # next to the weight ring, so K is split into windows whose partial sums
    # go through the workspace
    M, N, K = 4, 2048, 28672
    qc, qs = synth.weights(F4, N, K, 901)
    qx = synth.activations(M, K, 902)
    qc_d, qs_d, qx_d = dev_u8(qc), dev_u8(qs), dev_bf16(qx).view(M, K)
    # fused MoE down projection with the router-weighted combine
    T, E, topk, H, I = 4, 16, 4, 1024, 256
    dc, ds_ = synth.weights(F4, H, I, 903, E=E)
    h = synth.activations(T * topk, I, 904)
    ids = synth.expert_ids(T, E, topk, 905)
    r = synth.router_weights(T, topk, 906)
    dc_d, ds_d, h_d, ids_d = dev_u8(dc), dev_u8(ds_), dev_bf16(h).view(T * topk, I), dev_i32(ids)
    r_d = torch.from_numpy(r).cuda()
    # NVFP4 quantisation (tensor maximum through the workspace)
    XM, XK = 64, 4096
    xq = synth.activations(XM, XK, 907)
    xq_d = dev_bf16(xq).view(XM, XK)

    def run_all():
        y = ops.qmv(F4, qc_d, qs_d, qx_d, N)
        out = ops.moe_down_combine(F4, dc_d, ds_d, h_d, ids_d, r_d, E, H)
        c, s = ops.quantize(NV, xq_d)
        return y, out, c, s

    # a lone call on the default stream, anchored to the oracle
    y0, out0, c0, s0 = (t.cpu().numpy() for t in run_all())
    rows = np.arange(0, N, 37)
    check_close(y0[:, rows], orc.qmv_rows(F4, qc, qs, qx, M, N, K, rows), "qmv split-K")
    yd, rc = orc.moe_qmv(F4, dc, ds_, h, ids.reshape(-1, 1), T * topk, E, 1, H, I)
    assert rc == 0
    check_close(out0, orc.moe_combine(yd.reshape(T * topk, H), r, T, topk, H), "down-combine")
    wc, ws = orc.quantize(NV, xq, XM, XK)
    assert np.array_equal(c0, wc) and np.array_equal(s0, ws)

    failures = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                results = [run_all() for _ in range(ITERS)]
                stream.synchronize()
            for it, (y, out, c, s) in enumerate(results):
                same = (np.array_equal(y.cpu().numpy().view(np.uint32), y0.view(np.uint32))
                        and np.array_equal(out.cpu().numpy().view(np.uint32), out0.view(np.uint32))
                        and np.array_equal(c.cpu().numpy(), c0) and np.array_equal(s.cpu().numpy(), s0))
                if not same:
                    failures.append((i, it))
        except Exception as exc:  # reported below
            failures.append((i, repr(exc)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not failures, f"threads / iterations that differed from a lone call: {failures[:10]}"
    assert ops.device_error() == 0
