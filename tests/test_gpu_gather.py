"""Byte- and bit-exact checks of the decode path's page gather and of the
CUDA-core kernel's e4m3 dequant against the oracle's definitions: the
gather against the dense K[b, g, 0:L, :] / V[b, g, 0:L, :] rows read
through the block table on the host, in every KV layout; the dequant
against the oracle's 256-entry e4m3 table (NaN codes as NaN)."""

import numpy as np
import pytest
import torch

import oracle
import paged_fp8_kv_gb300 as mj
from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def dense_rows(w, cache, b, g):
    """K or V rows 0 .. L-1 of sequence b, kv head g: page block_table[b][j // PS], row j % PS."""
    L, PS = int(w.seq_lens[b]), w.page_size
    j = np.arange(L)
    return cache[w.block_table[b, j // PS], j % PS, g, :]


WORKLOADS = [
    ("tiny", lambda: syn.config(1)),
    ("edges_ps16", lambda: syn.make_workload("edges", [0, 1, 17, 128, 129, 300], 1, 2, 4, 16, seed=41)),
    ("gqa_ps16", lambda: syn.config(2, num_seqs=4, len_range=(1, 900))),
    ("spec_ps64", lambda: syn.config(4, num_seqs=3, len_range=(100, 700))),
    ("fp8_ps128", lambda: syn.config(3, num_seqs=3, len_range=(3000, 300), max_splits=16)),
    ("ps32", lambda: syn.make_workload("ps32", [31, 32, 33, 1000], 1, 3, 4, 32, seed=43)),
]


@pytest.mark.parametrize("layout", ["nhd", "hnd", "interleaved", "flashinfer"])
@pytest.mark.parametrize("name,make", WORKLOADS, ids=[x[0] for x in WORKLOADS])
def test_gather_is_byte_exact(name, make, layout):
    w = make()
    s = DecodeSession(w, kv_layout=layout)
    out_rows = max(128, -(-int(w.seq_lens.max()) // 128) * 128)
    for values in (False, True):
        out = torch.full((w.num_seqs, w.h_k, out_rows, 128), 0xEE, dtype=torch.uint8, device="cuda")
        mj.check_gather_kv(s.params, s.k_cache, s.v_cache, s.block_table, s.seq_lens, values, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        cache = w.v_cache if values else w.k_cache
        for b in range(w.num_seqs):
            L = int(w.seq_lens[b])
            for g in range(w.h_k):
                assert np.array_equal(got[b, g, :L], dense_rows(w, cache, b, g)), (name, layout, values, b, g)
                assert np.all(got[b, g, L:] == 0xEE)  # nothing written past the sequence end


def test_dequant_is_bit_exact():
    out = torch.full((256,), 7.0, dtype=torch.float32, device="cuda")
    mj.check_dequant_e4m3(out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.e4m3_table()
    for c in range(256):
        if np.isnan(ref[c]):
            assert np.isnan(got[c]), hex(c)
        else:
            assert got[c].view(np.uint32) == np.float32(ref[c]).view(np.uint32), hex(c)  # sign of zero too


@pytest.mark.parametrize("limit_us", [200, 2000])
def test_bounded_wait_gives_up_and_reports_a_timeout(limit_us):
    # the primitive every decode-kernel wait uses, on an mbarrier that never
    # completes: it must give up after its limit (not hang) and the status
    # word must read MJ_ERR_TIMEOUT; the GPU stays usable afterwards
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    mj.check_bounded_wait(status, waited, limit_us)
    torch.cuda.synchronize()
    assert int(status.item()) == mj.MJ_ERR_TIMEOUT
    ns = int(waited.item())
    assert limit_us * 1000 <= ns <= limit_us * 1000 + 5_000_000, ns
    # the context is intact: an ordinary launch still runs
    out = torch.empty(256, dtype=torch.float32, device="cuda")
    mj.check_dequant_e4m3(out)
    torch.cuda.synchronize()
    assert out[0].item() == 0.0
