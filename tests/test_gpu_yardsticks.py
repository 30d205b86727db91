"""The measurement yardsticks of the library on the GPU: pkv_hbm_copy (the
copy bandwidth the kernels are set against) copies bit-exactly and rejects
misaligned, ragged or overlapping ranges; pkv_hbm_gather_read (reads of
listed chunks, the decode's access pattern without its arithmetic) reads
exactly the listed chunks -- its XOR checksum equals one computed on the
CPU over the same words; pkv_fp32_fma_peak (the CUDA cores' fp32 rate) runs
every chain to the exact value a = b = 1 gives, plain and paired."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_67_gb300 as pkv

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.mark.parametrize("nbytes", [16, 4096, 1 << 20, (1 << 26) + 48])
def test_copy_is_bit_exact(nbytes):
    g = torch.Generator().manual_seed(nbytes % 1000)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).to(DEV)
    dst = torch.zeros_like(src)
    pkv.pkv_hbm_copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)


def test_copy_rejects_bad_ranges():
    lib = pkv.load_library()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.pkv_hbm_copy(ctypes.c_void_p(p + 4096), ctypes.c_void_p(p), 4008, s) == 1  # size % 16
    assert lib.pkv_hbm_copy(ctypes.c_void_p(p + 4104), ctypes.c_void_p(p), 4096, s) == 1  # dst alignment
    assert lib.pkv_hbm_copy(ctypes.c_void_p(p + 1024), ctypes.c_void_p(p), 4096, s) == 1  # overlap
    assert lib.pkv_hbm_copy(ctypes.c_void_p(p + 4096), ctypes.c_void_p(p), 0, s) == 0


def _xor_fold(words: np.ndarray) -> int:
    pairs = words.reshape(-1, 2)
    x = np.bitwise_xor.reduce(pairs[:, 0] ^ pairs[:, 1]) if pairs.size else np.uint64(0)
    return int(x)


@pytest.mark.parametrize("chunk_bytes,stride", [(32768, 32768), (4096, 32768), (4112, 8192), (16, 16)])
def test_gather_reads_exactly_the_listed_chunks(chunk_bytes, stride):
    g = torch.Generator().manual_seed(chunk_bytes + stride)
    nchunks_pool = 300
    pool = torch.randint(-2**62, 2**62, (nchunks_pool * stride // 8 + chunk_bytes // 8,),
                         dtype=torch.int64, generator=g)
    idx = torch.randperm(nchunks_pool, generator=g)[:257].to(torch.int32)
    want = 0
    words = pool.numpy().view(np.uint64)
    for i in idx.tolist():
        want ^= _xor_fold(words[i * stride // 8:(i * stride + chunk_bytes) // 8])
    sink = torch.zeros(1, dtype=torch.int64, device=DEV)
    pkv.pkv_hbm_gather_read(pool.to(DEV), idx.to(DEV), stride, chunk_bytes, sink)
    torch.cuda.synchronize()
    assert int(sink.cpu().numpy().view(np.uint64)[0]) == want


@pytest.mark.parametrize("paired", [False, True])
@pytest.mark.parametrize("iters", [0, 1, 1000, 4097])
def test_fma_chains_run_to_their_exact_value(paired, iters):
    """x <- x * 1 + 1 from 0 is exactly iters after iters steps (iters <
    2^24); thread 0 of every block stores the sum of its chains."""
    out = torch.full((37,), -5.0, dtype=torch.float32, device=DEV)
    pkv.pkv_fp32_fma_peak(out, iters, 1.0, 1.0, never=-1.0, paired=paired)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), torch.full((37,), float(pkv.FMA_CHAINS * iters)))


def test_fma_other_values_and_bad_args():
    """a = 0.5, b = 1: a chain converges to 2 - 2^-iters (exact in fp32
    for small iters); bad arguments are rejected before any launch."""
    out = torch.zeros(4, dtype=torch.float32, device=DEV)
    pkv.pkv_fp32_fma_peak(out, 10, 0.5, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), torch.full((4,), pkv.FMA_CHAINS * (2.0 - 2.0 ** -9)))
    lib = pkv.load_library()
    s = torch.cuda.current_stream().cuda_stream
    p = out.data_ptr()
    assert lib.pkv_fp32_fma_peak(ctypes.c_void_p(0), 4, 10, 1.0, 1.0, -1.0, 0, s) == 1
    assert lib.pkv_fp32_fma_peak(ctypes.c_void_p(p + 2), 1, 10, 1.0, 1.0, -1.0, 0, s) == 1
    assert lib.pkv_fp32_fma_peak(ctypes.c_void_p(p), 0, 10, 1.0, 1.0, -1.0, 0, s) == 1
    assert lib.pkv_fp32_fma_peak(ctypes.c_void_p(p), 4, -1, 1.0, 1.0, -1.0, 0, s) == 1


def test_gather_pair_reads_both_buffers_in_one_launch():
    """The pair gather's checksum is the XOR of the two single gathers'."""
    g = torch.Generator().manual_seed(7)
    stride = chunk = 4096
    a = torch.randint(-2**62, 2**62, (200 * stride // 8,), dtype=torch.int64, generator=g)
    b = torch.randint(-2**62, 2**62, (200 * stride // 8,), dtype=torch.int64, generator=g)
    idx = torch.randperm(200, generator=g)[:77].to(torch.int32)
    wa, wb = a.numpy().view(np.uint64), b.numpy().view(np.uint64)
    want = 0
    for i in idx.tolist():
        want ^= _xor_fold(wa[i * stride // 8:(i * stride + chunk) // 8])
        want ^= _xor_fold(wb[i * stride // 8:(i * stride + chunk) // 8])
    sink = torch.zeros(1, dtype=torch.int64, device=DEV)
    pkv.pkv_hbm_gather_read_pair(a.to(DEV), b.to(DEV), idx.to(DEV), stride, chunk, sink)
    torch.cuda.synchronize()
    assert int(sink.cpu().numpy().view(np.uint64)[0]) == want
