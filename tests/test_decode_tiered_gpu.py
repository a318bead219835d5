"""GPU parity of attn_decode_tiered (a cold cache -- contiguous or paged, f16 or
int8 -- plus an f16 hot ring, one softmax over both) against the oracle,
through the C ABI: ragged tiers, empty tiers, rings that have overwritten their
oldest hot tokens, rings starting mid-way, windows ending in either tier, and
the bit-identity with attn_decode when the hot tier is empty."""
import numpy as np
import pytest
import torch

import attention_split_kv_gb300 as attn
import oracle
import seeded_inputs as si
from parity_util import assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    attn.build()
    attn.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    yield
    assert attn.attn_device_status() == attn.ATTN_OK


def _run(case, split_keys=0):
    g = case.to("cuda")
    lse = torch.empty((case.batch, case.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode_tiered(g, lse_out=lse, split_keys=split_keys)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(case, what, split_keys=0):
    ref, ref_lse = oracle.decode_tiered(case)
    got, lse = _run(case, split_keys)
    assert_close(got.reshape(ref.shape), ref, int8=case.int8, what=what)
    assert_lse_close(lse.reshape(-1), ref_lse, what=what)


LENS = dict(cold=[0, 300, 17, 1000, 64], hot=[0, 40, 200, 5, 64])   # 200 > ring: overwritten


@pytest.mark.parametrize("int8,page_size", [(False, 0), (False, 16), (False, 8), (True, 0), (True, 16)],
                         ids=["f16", "f16_paged16", "f16_paged8", "int8", "int8_paged16"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_tiered_matches_oracle(int8, page_size, D):
    c = si.make_tiered_case(5, 8, 2, D, LENS["cold"], LENS["hot"], 64, seed=D + page_size + int8,
                            int8=int8, page_size=page_size)
    _check(c, "tiered D=%d int8=%s P=%d" % (D, int8, page_size))


@pytest.mark.parametrize("window", [1, 30, 100, 500])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
def test_tiered_window_across_the_tiers(window, int8):
    # windows ending inside the hot ring (1, 30), just past it (100) and deep in the cold tier
    c = si.make_tiered_case(5, 8, 2, 128, LENS["cold"], LENS["hot"], 64, seed=window, int8=int8, page_size=16,
                            window=window)
    _check(c, "tiered window %d" % window)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (6, 2), (32, 8)])
def test_tiered_gqa_and_softcap(Hq, Hkv):
    c = si.make_tiered_case(3, Hq, Hkv, 128, [123, 0, 999], [77, 33, 0], 96, seed=Hq, page_size=32,
                            softcap=30.0)
    _check(c, "tiered GQA %d/%d" % (Hq, Hkv))


@pytest.mark.parametrize("split_keys", [16, 64, 0])
def test_tiered_splits(split_keys):
    c = si.make_tiered_case(4, 32, 8, 128, (500, 3000), (100, 1024), 1024, seed=9, page_size=16)
    _check(c, "tiered split %d" % split_keys, split_keys)


@pytest.mark.parametrize("int8,page_size", [(False, 16), (True, 0), (False, 8)])
def test_tiered_without_hot_tokens_is_bit_identical_to_decode(int8, page_size):
    # an empty hot tier contributes no item to the combine: the cold tier's split
    # plan and arithmetic order are attn_decode's
    c = si.make_tiered_case(4, 8, 2, 128, [1, 200, 777, 64], [0, 0, 0, 0], 32, seed=5, int8=int8,
                            page_size=page_size, window=300)
    cold = si.DecodeCase(**{k: v for k, v in c.__dict__.items() if k in si.DecodeCase.__dataclass_fields__})
    a, la = _run(c, split_keys=64)
    g = cold.to("cuda")
    lse = torch.empty((4, 8), dtype=torch.float32, device="cuda")
    b = attn.decode(g, lse_out=lse, split_keys=64).float().cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(a, b) and np.array_equal(la, lse.cpu().numpy())


def test_tiered_rejects_bad_hot_ring():
    c = si.make_tiered_case(1, 4, 2, 64, [10], [5], 16, seed=3).to("cuda")
    out = torch.empty((1, 4, 64), dtype=torch.float16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in (0, 8, 40):
        with pytest.raises(attn.AttnError) as e:
            attn.attn_decode_tiered(c.q, attn.ATTN_F16, c.k, c.v, None, None, attn.ATTN_KV_F16, c.kv_len, None, 0, 0,
                                    0, c.cap, c.hot_k, c.hot_v, c.hot_len, c.hot_start, bad, 1, 4, 2, 64, 0, 0.0,
                                    0.125, 0, out, attn.ATTN_F16, None, ws, ws.numel())
        assert e.value.status == attn.ATTN_EUNSUPPORTED
