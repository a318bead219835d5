"""GPU parity of attn_decode_ring (decode over a ring / rolling-buffer KV
cache, token t in slot t % ring) against the oracle, and against attn_decode
on the contiguous cache holding the same logical tokens with the ring's
effective window.  Unwritten ring slots hold filler values that no result may
depend on."""
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


def _run(case, split_keys=0, max_kv=None):
    g = case.to("cuda")
    lse = torch.empty((case.batch, case.n_heads), dtype=torch.float32, device="cuda")
    out = attn.decode(g, lse_out=lse, split_keys=split_keys, max_kv=max_kv)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _ring_case(B, Hq, Hkv, D, lens, ring, window, int8, seed, softcap=0.0):
    cc = si.make_decode_case(B, Hq, Hkv, D, lens, seed=seed, int8=int8, window=window, softcap=softcap)
    return cc, si.ring_from_contiguous(cc, ring)


RING_SHAPES = [
    # B, Hq, Hkv, D, lens, ring, window
    (4, 8, 2, 128, [1, 100, 256, 1000], 256, 0),       # shorter than, equal to and 4x the ring
    (3, 8, 2, 128, [37, 517, 2049], 128, 100),         # window inside the ring, ragged starts
    (3, 8, 2, 128, [37, 517, 2049], 128, 500),         # window wider than the ring: the ring wins
    (2, 4, 2, 64, [33, 700], 64, 0),                   # D=64
    (2, 6, 2, 64, [250, 17], 48, 0),                   # G=3, ring not a power of two
    (2, 16, 2, 256, [500, 129], 96, 0),                # D=256 (CUDA-core kernel)
    (2, 8, 8, 128, [300, 4096], 512, 0),               # MHA, long logical length
    (3, 8, 2, 128, [0, 16, 17], 16, 0),                # empty sequence, one-tile ring
]


# split_keys 0: the automatic plan (rings of at most 512 slots run the one-launch
# direct kernel); 16 forces the split path, whose splits cross the ring's seam
@pytest.mark.parametrize("split_keys", [0, 16], ids=["auto", "split16"])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("shape", RING_SHAPES, ids=lambda s: "B%d_H%d_%d_D%d_R%d_W%d" % (s[:4] + s[5:]))
def test_ring_decode_matches_oracle(shape, int8, split_keys):
    B, Hq, Hkv, D, lens, ring, window = shape
    _, rc = _ring_case(B, Hq, Hkv, D, lens, ring, window, int8, seed=ring + D + window)
    ref, ref_lse = oracle.decode(rc)
    got, lse = _run(rc, split_keys=split_keys)
    assert_close(got.reshape(ref.shape), ref, int8=int8, what="ring %s" % (shape,))
    assert_lse_close(lse.reshape(-1), ref_lse, what="ring %s" % (shape,))


@pytest.mark.parametrize("split_keys", [16, 64, 0])
def test_ring_decode_splits(split_keys):
    # many splits per sequence, split boundaries that cross the ring's seam
    _, rc = _ring_case(4, 32, 8, 128, [5, 1500, 3001, 777], 1024, 0, False, seed=77)
    ref, ref_lse = oracle.decode(rc)
    got, lse = _run(rc, split_keys=split_keys)
    assert_close(got.reshape(ref.shape), ref, int8=False, what="ring split %d" % split_keys)
    assert_lse_close(lse.reshape(-1), ref_lse, what="ring split %d" % split_keys)


def test_ring_decode_softcap():
    _, rc = _ring_case(2, 8, 2, 128, [90, 1000], 64, 40, False, seed=5, softcap=30.0)
    ref, ref_lse = oracle.decode(rc)
    got, lse = _run(rc)
    assert_close(got.reshape(ref.shape), ref, int8=False, what="ring softcap")
    assert_lse_close(lse.reshape(-1), ref_lse, what="ring softcap")


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("ring,window", [(64, 0), (128, 50), (32, 1000)])
def test_ring_equals_contiguous_with_window(ring, window, int8):
    # the ring keeps the last min(L, ring, W) tokens: attn_decode on the
    # contiguous cache with that window computes the same attention
    cc, rc = _ring_case(3, 8, 2, 128, [20, 333, 1200], ring, window, int8, seed=11)
    w_eff = ring if window <= 0 else min(window, ring)
    cw = si.DecodeCase(**{**cc.__dict__, "window": w_eff})
    a, la = _run(cw, split_keys=64)
    b, lb = _run(rc, split_keys=64)
    np.testing.assert_allclose(b, a, rtol=0, atol=2e-3)
    np.testing.assert_allclose(lb, la, rtol=0, atol=1e-4)


def test_ring_rejects_bad_ring_size():
    _, rc = _ring_case(1, 4, 2, 64, [10], 16, 0, False, seed=3)
    g = rc.to("cuda")
    out = torch.empty((1, 4, 64), dtype=torch.float16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in (0, 8, 24, -16):
        with pytest.raises(attn.AttnError) as e:
            attn.attn_decode_ring(g.q, g.k, g.v, g.kv_len, bad, None, None, attn.ATTN_KV_F16, 1, 4, 2, 64,
                                  0, 0.0, 0.125, 0, out, None, ws, ws.numel())
        assert e.value.status == attn.ATTN_EUNSUPPORTED
