"""GPU checks of the measurement helpers behind the roofline denominators:
the memory-stream probe (mm_stream_probe) writes and copies exactly what it
claims, and the arithmetic-rate probe (mm_alu_probe) runs the stated number of
dependent multiply-adds (its int32 chains are recomputed on the host)."""

import numpy as np
import pytest
import torch

import quantized_gemm_gb300 as qg

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_stream_probe_write_and_copy():
    n = (8 << 20) + 48
    dst = torch.zeros(n, dtype=torch.uint8, device=DEV)
    for mode in (0, 2):
        dst.zero_()
        qg.mm_stream_probe(dst, None, mode)
        torch.cuda.synchronize()
        got = dst.cpu().numpy()
        if mode == 0:
            assert np.all(got.view(np.uint32) == 0x3f803f80)
        else:
            assert np.all(got == 0)
    src = torch.randint(0, 256, (n,), dtype=torch.uint8, device=DEV)
    qg.mm_stream_probe(dst, src, 1)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)


def test_alu_probe_int32_chains():
    iters = 7
    macs = qg.mm_alu_probe(0, iters)
    chains = qg.MM_ALU_CHAINS
    threads = macs // (chains * iters)
    assert threads > 0 and macs == threads * chains * iters
    out = torch.zeros(threads, dtype=torch.int64, device=DEV)
    qg.mm_alu_probe(0, iters, out=out)
    torch.cuda.synchronize()
    # one 32-bit sum per thread, packed at the start of the buffer
    got = out.cpu().numpy().view(np.uint32)[:threads]
    seed = (iters * 2654435761) & 0xFFFFFFFF
    a, c = seed | 1, seed ^ 0x9E3779B9
    tid = np.arange(threads, dtype=np.uint64)
    s = np.zeros(threads, dtype=np.uint64)
    for j in range(chains):
        x = (tid + j) & 0xFFFFFFFF
        for _ in range(iters):
            x = (x * a + c) & 0xFFFFFFFF
        s = (s + x) & 0xFFFFFFFF
    assert np.array_equal(got.astype(np.uint64), s)


@pytest.mark.parametrize("op", [1, 2])
def test_alu_probe_float_chains_run(op):
    iters = 50
    macs = qg.mm_alu_probe(op, iters)
    out = torch.zeros(macs // (qg.MM_ALU_CHAINS * iters), dtype=torch.float64, device=DEV)
    qg.mm_alu_probe(op, iters, out=out)
    torch.cuda.synchronize()
    threads = macs // (qg.MM_ALU_CHAINS * iters)
    vals = out if op == 1 else out.view(torch.float32)[:threads]   # fp32 sums are packed
    assert torch.isfinite(vals).all() and (vals != 0).any()
    with pytest.raises(qg.MMError):
        qg.mm_alu_probe(7, iters)
