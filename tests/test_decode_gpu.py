"""GPU parity of attn_decode (split-KV decode + LSE combine) against the oracle,
through the C ABI, on seeded inputs spanning several tiles, splits and ragged
tails."""
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


def _run(case, split_keys=0, max_kv=None, with_lse=True):
    g = case.to("cuda")
    lse = torch.empty((case.batch, case.n_heads), dtype=torch.float32, device="cuda") if with_lse else None
    out = attn.decode(g, lse_out=lse, split_keys=split_keys, max_kv=max_kv)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)


def _check(case, split_keys=0, max_kv=None, what=""):
    ref, ref_lse = oracle.decode(case)
    got, lse = _run(case, split_keys, max_kv)
    assert_close(got.reshape(ref.shape), ref, int8=case.int8, what=what)
    assert_lse_close(lse.reshape(-1), ref_lse, what=what)
    return got


SHAPES = [
    # B, Hq, Hkv, D, lens
    (1, 4, 2, 64, [128]),                 # the tiny GQA 2:1 decode
    (3, 8, 2, 128, [1, 77, 1000]),        # G=4, ragged tails, one single-token sequence
    (2, 8, 8, 128, [300, 33]),            # MHA (G=1)
    (2, 6, 2, 64, [250, 17]),             # G=3 -> three single-head groups
    (2, 16, 2, 256, [500, 129]),          # D=256, G=8 -> two 4-head groups
    (2, 4, 2, 256, [64, 1]),
]


# split_keys 0 is the automatic plan (the one-launch direct kernel for the shapes
# whose sequences keep at most 512 keys); 16 forces the split path
@pytest.mark.parametrize("split_keys", [0, 16], ids=["auto", "split16"])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%d_H%d_%d_D%d" % s[:4])
def test_decode_contiguous(shape, int8, split_keys):
    B, Hq, Hkv, D, lens = shape
    case = si.make_decode_case(B, Hq, Hkv, D, lens, seed=hash((B, Hq, D)) % 1000, int8=int8)
    _check(case, split_keys=split_keys, what="contiguous %s split %d" % (shape, split_keys))


@pytest.mark.parametrize("page_size", [1, 8, 16, 64])
@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
def test_decode_paged(page_size, int8):
    if int8 and page_size < 8:
        pytest.skip("int8 caches need pages of >= 8 tokens")
    case = si.make_decode_case(4, 8, 2, 128, (1, 700), seed=31 + page_size, int8=int8,
                               page_size=page_size)
    _check(case, what="paged P=%d" % page_size)


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("page_size", [1, 2, 4, 8, 16, 32])
def test_paged_is_bit_identical_to_contiguous(page_size, int8):
    # the page table only changes where rows are read from: both layouts run the
    # same kernel and give the same bits.  int8 caches run the CUDA-core kernel
    # for every layout.  Here (8 query / 2 kv heads, D=128) an f16 TMA box spans
    # NH=2 kv heads; the tensor-core kernel takes pages of 16k tokens, and pages
    # of P tokens with P * NH >= 8 (P >= 4), each box of P rows starting
    # 1024-byte aligned.  Shorter f16 pages run the CUDA-core kernel while the
    # contiguous cache runs the tensor-core one: there the two agree to the
    # parity tolerance; the tests below pin bit-identity for those page sizes
    # where one kernel runs both.
    if int8 and page_size < 8:
        pytest.skip("int8 caches need pages of >= 8 tokens")
    case = si.make_decode_case(3, 8, 2, 128, [5, 450, 300], seed=41, int8=int8, cap=456)
    paged = si.paged_from_contiguous(case, page_size, seed=42)
    a, la = _run(case, split_keys=64, max_kv=456)
    b, lb = _run(paged, split_keys=64, max_kv=456)
    same_kernel = int8 or page_size % 16 == 0 or page_size * 2 >= 8
    if same_kernel:
        assert np.array_equal(a, b) and np.array_equal(la, lb)
    else:
        assert np.abs(a - b).max() <= 2e-3 and np.abs(la - lb).max() <= 1e-3


@pytest.mark.parametrize("page_size", [1, 2, 8])
def test_one_token_pages_bit_identical_on_the_tensor_core_kernel(page_size):
    # 32 query / 8 kv heads: a box spans NH=8 kv heads, so even 1-token pages
    # start every box 1024-byte aligned and run the tensor-core kernel
    case = si.make_decode_case(3, 32, 8, 128, [5, 450, 300], seed=43, cap=456)
    paged = si.paged_from_contiguous(case, page_size, seed=44)
    a, la = _run(case, split_keys=64, max_kv=456)
    b, lb = _run(paged, split_keys=64, max_kv=456)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("int8", [False, True], ids=["f16", "int8"])
@pytest.mark.parametrize("page_size", [1, 8, 16])
def test_paged_bit_identical_on_the_cuda_core_kernel(page_size, int8):
    # D=256 runs the CUDA-core kernel for both layouts, whatever the page size
    if int8 and page_size < 8:
        pytest.skip("int8 caches need pages of >= 8 tokens")
    case = si.make_decode_case(3, 8, 2, 256, [5, 450, 300], seed=45, int8=int8, cap=456)
    paged = si.paged_from_contiguous(case, page_size, seed=46)
    a, la = _run(case, split_keys=64, max_kv=456)
    b, lb = _run(paged, split_keys=64, max_kv=456)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("window", [1, 5, 16, 100, 5000])
def test_decode_sliding_window(window):
    case = si.make_decode_case(3, 8, 2, 128, [50, 333, 1200], seed=51, window=window)
    _check(case, what="window %d" % window)
    paged = si.make_decode_case(3, 8, 2, 64, [50, 333, 1200], seed=52, window=window, page_size=16,
                                int8=True)
    _check(paged, what="paged int8 window %d" % window)


@pytest.mark.parametrize("softcap", [1.0, 30.0])
def test_decode_softcap(softcap):
    case = si.make_decode_case(2, 8, 2, 128, [400, 90], seed=61, softcap=softcap, scale=0.3)
    _check(case, what="softcap %g" % softcap)


@pytest.mark.parametrize("split_keys", [16, 48, 112, 256, 4096])
def test_split_count_does_not_change_the_result(split_keys):
    case = si.make_decode_case(2, 8, 2, 128, [1000, 217], seed=71)
    got = _check(case, split_keys=split_keys, what="split %d" % split_keys)
    base, _ = _run(case, split_keys=0)
    assert np.abs(got - base).max() <= 2e-3


@pytest.mark.parametrize("B", [2048, 2049, 4096])
def test_decode_largest_batches(B):
    # 2048 sequences is the tensor-core kernel's limit (its prefixes live in shared
    # memory); 2049 falls back to the CUDA-core kernel; 4096 is the library's limit
    # (an explicit split size keeps these small sequences on the split path)
    lens = [(7 * b) % 61 for b in range(B)]   # 0 .. 60 keys, some empty
    case = si.make_decode_case(B, 8, 2, 64, lens, seed=B, page_size=16)
    ref, ref_lse = oracle.decode(case)
    got, lse = _run(case, split_keys=16)
    assert_close(got.reshape(ref.shape), ref, what="batch %d" % B)
    assert_lse_close(lse.reshape(-1), ref_lse, what="batch %d" % B)


@pytest.mark.parametrize("split_keys", [0, 16], ids=["auto", "split16"])
def test_zero_length_sequence(split_keys):
    case = si.make_decode_case(3, 4, 2, 64, [0, 20, 0], seed=81, cap=32)
    got, lse = _run(case, split_keys=split_keys)
    got = got.reshape(3, 4, 64)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert np.all(np.isneginf(lse[0])) and np.all(np.isneginf(lse[2]))
    ref, _ = oracle.decode(case)
    assert_close(got.reshape(ref.shape)[4:8], ref[4:8], what="zero-length neighbours")


@pytest.mark.parametrize("split_keys", [0, 16], ids=["auto", "split16"])
def test_kv_len_above_capacity_is_clamped_not_faulting(split_keys):
    case = si.make_decode_case(2, 4, 2, 64, [40, 64], seed=91, cap=64)
    big = case.to("cuda")
    big.kv_len = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    out = attn.decode(big, split_keys=split_keys)
    torch.cuda.synchronize()
    ref, _ = oracle.decode(case)      # same as kv_len clamped to the capacity (64)
    assert_close(out.float().cpu().numpy().reshape(ref.shape), ref, what="clamped")
    st, bad = attn.attn_decode_validate(big.kv_len, None, 2, 0, 0, 0, 64)
    assert st == attn.ATTN_EBOUNDS and bad == 1


def test_validate_entry_point():
    case = si.make_decode_case(3, 4, 2, 64, [40, 17, 100], seed=93, page_size=16).to("cuda")
    args = (case.batch, case.page_size, case.max_pages, case.n_pages, case.cap)
    assert attn.attn_decode_validate(case.kv_len, case.page_table, *args)[0] == attn.ATTN_OK
    pt = case.page_table.clone()
    pt[2, 3] = case.n_pages + 5           # a page the sequence uses, out of the pool
    st, bad = attn.attn_decode_validate(case.kv_len, pt, *args)
    assert st == attn.ATTN_EBOUNDS and bad == 2
    pt = case.page_table.clone()
    pt[1, 5] = -7                         # past sequence 1's pages (17 tokens = 2 pages): unused
    assert attn.attn_decode_validate(case.kv_len, pt, *args)[0] == attn.ATTN_OK
    kl = case.kv_len.clone()
    kl[0] = 0
    st, bad = attn.attn_decode_validate(kl, case.page_table, *args)
    assert st == attn.ATTN_EINVAL and bad == 0


@pytest.mark.parametrize("split_keys", [0, 16], ids=["auto", "split16"])
def test_invalid_page_id_is_replaced_and_reported(split_keys):
    # the kernel checks every page id it uses against the pool: an id outside
    # it is replaced by page 0 (never read out of bounds) and reported
    case = si.make_decode_case(2, 4, 2, 64, [40, 30], seed=95, page_size=16).to("cuda")
    case.page_table = case.page_table.clone()
    case.page_table[0, 1] = 10_000_000
    out = attn.decode(case, split_keys=split_keys)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert attn.attn_device_status() == attn.ATTN_EBOUNDS
    assert attn.attn_device_status() == attn.ATTN_OK      # the report clears the word
    ref, _ = oracle.decode(case.to("cpu"))
    assert_close(out.float().cpu().numpy().reshape(ref.shape)[4:], ref[4:], what="other sequence")


def test_repeated_calls_reuse_workspace_without_clearing():
    case = si.make_decode_case(4, 8, 2, 128, (100, 900), seed=97, page_size=16)
    g = case.to("cuda")
    ws = torch.full((attn.attn_decode_workspace_size(4, 8, 2, 128, g.cap),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    a = attn.decode(g, workspace=ws).clone()
    b = attn.decode(g, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
