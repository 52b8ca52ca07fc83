"""Several host threads calling the library at once, each on its own stream.

The per-device state (properties, memory pool, tensor-map encoder, the host-buffer calls'
copy streams, the softmax launch state) is created under locks on first use; the test starts
every thread before any of them has called the library, so the first calls race, and checks
that each thread's results equal those of a single-threaded run bit for bit (the same
kernels on the same inputs).
"""
import threading

import numpy as np
import pytest

import tensor_core_tiled_gb300 as tct

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _work(seed, stream):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(300, 150, device="cuda", generator=g).half()        # repacked (lda = 150)
    B = torch.randn(150, 200, device="cuda", generator=g).half()
    A2 = torch.randn(1024, 1024, device="cuda", generator=g).half()
    X = torch.randn(1000, 3000, device="cuda", generator=g)
    hA = torch.randn(700, 300, generator=torch.Generator().manual_seed(seed)).half().pin_memory()
    hB = torch.randn(300, 500, generator=torch.Generator().manual_seed(seed + 1)).half().pin_memory()
    hC = torch.empty(700, 500).pin_memory()
    with torch.cuda.stream(stream):
        outs = [tct.matmul(A, B), tct.matmul(A2, A2), tct.softmax(X)]
        st = tct.gemm_f16_f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), 700, 500, 300, 300, 500, 500,
                                   stream.cuda_stream)
        assert st == tct.GEMM_OK
    stream.synchronize()
    return [o.cpu().numpy() for o in outs] + [hC.numpy().copy()]


def test_concurrent_threads_match_single_threaded(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    seeds = [11, 12, 13, 14]
    results, errors = {}, []
    start = threading.Barrier(len(seeds))

    def run(seed):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            start.wait()
            results[seed] = [_work(seed, s) for _ in range(3)]
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(sd,)) for sd in seeds]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK
    for seed in seeds:
        ref = _work(seed, torch.cuda.Stream())
        for rep in results[seed]:
            for got, want in zip(rep, ref):
                assert np.array_equal(got.view(np.int32), want.view(np.int32))
