"""The failure path of the kernels' bounded waits, on the GPU, without a fault.

The testing hook shortens the pipeline-wait limit to 20 ms and makes one wait
of every CTA run out: the tensor-core kernels hold back the signal of their
first S tile, the CUDA-core decode kernel issues no copy.  A wait that runs out
records a code in the library's device error word, raises the CTA's abort flag,
lets the copies and tensor-core work already in flight land, frees the CTA's
tensor memory and returns.  Each case checks that the call returns, that
attn_device_status reports ATTN_ETIMEOUT (and clears it), and that the next
normal call on the same context passes parity: its TMEM allocation would wait
forever had the aborted kernel kept its columns."""
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import assert_close

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    assert attn.attn_device_status() == attn.ATTN_OK
    yield
    assert attn.attn_testing_set_waits(0, 0) == attn.ATTN_OK
    assert attn.attn_device_status() == attn.ATTN_OK


def _stalled(call):
    assert attn.attn_testing_set_waits(LIMIT_NS, 1) == attn.ATTN_OK
    try:
        call()
        st = attn.attn_device_status()          # synchronises
    finally:
        assert attn.attn_testing_set_waits(0, 0) == attn.ATTN_OK
    return st


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_timeout_reports_and_recovers(D):
    pc = si.make_prefill_case(300, 4, 2, D, seed=D, causal=True)
    g = pc.to("cuda")
    assert _stalled(lambda: attn.prefill(g)) == attn.ATTN_ETIMEOUT
    assert attn.attn_device_status() == attn.ATTN_OK          # the report cleared the word
    ref, _ = oracle.prefill(pc)
    out = attn.prefill(g)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, what="after timeout D=%d" % D)


@pytest.mark.parametrize("kind", ["tensor_core_f16", "cuda_core_int8", "cuda_core_d256"])
def test_decode_timeout_reports_and_recovers(kind):
    # f16 with D=128 and 16-token pages runs the tensor-core kernel; int8 caches
    # and D=256 run the CUDA-core kernel
    int8 = kind == "cuda_core_int8"
    D = 256 if kind == "cuda_core_d256" else 128
    case = si.make_decode_case(3, 8, 2, D, [700, 33, 1000], seed=11, int8=int8, page_size=16)
    g = case.to("cuda")
    assert _stalled(lambda: attn.decode(g)) == attn.ATTN_ETIMEOUT
    ref, _ = oracle.decode(case)
    out = attn.decode(g)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, int8=int8, what="after timeout " + kind)


def test_hook_rejects_bad_values_and_restores_defaults():
    assert attn.attn_testing_set_waits(0, 2) == attn.ATTN_EINVAL
    assert attn.attn_testing_set_waits(0, 0) == attn.ATTN_OK
