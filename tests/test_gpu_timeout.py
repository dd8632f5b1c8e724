"""Failure detection on the GPU without a fault: a pipeline barrier that never
completes makes the bounded wait on it run out; the kernel records the
timeout, lets its copies land and returns, nvfp4_sync_check reports
NVFP4_ERR_TIMEOUT once, and the device keeps working (the next calls are
bit-identical to the calls made before the timeout)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import nvfp4_bit_block_02_b300 as nv

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms
TIMEOUT = 5


def _bf16(rows, cols, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.standard_normal((rows, cols)).astype(np.float32)).to(torch.bfloat16).cuda()


def _expect_timeout():
    with pytest.raises(nv.NVFP4Error) as e:
        nv.sync_check()
    assert e.value.status == TIMEOUT
    nv.sync_check()  # reported once: the word was cleared by the exchange


def _same(q1, q2):
    assert torch.equal(q1.codes, q2.codes) and torch.equal(q1.scales, q2.scales)
    assert torch.equal(q1.amax, q2.amax) and torch.equal(q1.global_scale, q2.global_scale)


@pytest.mark.parametrize("rht", [False, True])
def test_transposed_encoder_wait_runs_out(rht):
    x = _bf16(512, 1024, 11)

    def run():
        if rht:
            return nv.rht_quantize(x, rht_seed=3, rounding="stochastic", seed=5)[0]
        return nv.quantize(x, transpose=True)

    before = run()
    nv.sync_check()
    try:
        nv.test_expire_next_wait(nv.TEST_TRANSPOSED_ENCODER, LIMIT_NS)
        run()  # outputs undefined
    finally:
        nv.test_expire_next_wait(nv.TEST_TRANSPOSED_ENCODER, 0)
    _expect_timeout()
    after = run()
    nv.sync_check()
    _same(before, after)


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (512, 768, 1024)])
def test_gemm_wait_runs_out(M, N, K):
    qa = nv.quantize(_bf16(M, K, M + K))
    qb = nv.quantize(_bf16(N, K, N + K), block="2d")
    before = nv.gemm(qa, qb)
    nv.sync_check()
    try:
        nv.test_expire_next_wait(nv.TEST_GEMM, LIMIT_NS)
        nv.gemm(qa, qb)  # output undefined
    finally:
        nv.test_expire_next_wait(nv.TEST_GEMM, 0)
    _expect_timeout()
    after = nv.gemm(qa, qb)
    nv.sync_check()
    assert torch.equal(before, after)
    # the other GEMM variants are not armed and run normally
    d, _ = nv.gemm_amax(qa, qb)
    nv.sync_check()
    assert torch.equal(d, before)
