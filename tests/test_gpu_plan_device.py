"""The device-side plan (mj_decode_plan_device): bit-exact against the host
plan and the oracle's restatement for the same options, its status word,
and a CUDA graph of (device plan, decode, merge) replayed with changing
sequence lengths, checked against the fp64 oracle at every replay."""

import dataclasses

import numpy as np
import pytest
import torch

import paged_fp8_kv_gb300 as mj
from oracle.plan_ref import plan_ref
from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def device_plan(p, lens, pad_to, **opts):
    sl = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    work = torch.full((pad_to, 4), -7, dtype=torch.int32, device="cuda")
    ns = torch.full((len(lens),), -7, dtype=torch.int32, device="cuda")
    chunk = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    used = mj.decode_plan_device(p, sl, work, ns, pad_to, chunk_tiles=chunk, status=status, **opts)
    torch.cuda.synchronize()
    return used, work.cpu().numpy(), ns.cpu().numpy(), int(chunk.item()), int(status.item())


def test_matches_host_plan_and_oracle_on_random_workloads():
    rng = np.random.default_rng(2024)
    for trial in range(150):
        b = int(rng.integers(1, 300))
        h_k = int(rng.choice([1, 2, 8]))
        q_len = int(rng.choice([1, 4]))
        h_r = int(rng.choice([4, 8, 16]))
        ps = int(rng.choice([16, 128]))
        maxlen = int(rng.choice([1000, 16384, 131072]))
        lens = rng.integers(0, maxlen + 1, size=b).astype(np.int32)
        if rng.random() < 0.25:
            lens[:] = maxlen
        if rng.random() < 0.2:
            lens[rng.integers(0, b)] = 0
        mb = (maxlen + ps - 1) // ps
        ms = int(rng.choice([1, 16, 64, 256]))
        p = mj.make_params(b, q_len, h_k, h_r, ps, mb, b * mb, True, mj.MJ_BF16, ms, 128, int(rng.choice([0, 2])), 0)
        cps = int(rng.choice([0, 1, 3, 5, 24]))
        force = int(rng.choice([0, 0, 0, 2, 7])) if ms > 1 else 0
        minc = int(rng.choice([0, 0, 3]))
        pad_to = b * ms
        used, work, ns, chunk, status = device_plan(
            p, lens, pad_to, sm_count=152, ctas_per_sm=cps, force_splits=force, min_chunk_tiles=minc
        )
        # the host plan with the options the device plan resolved (explicit
        # ctas_per_sm: no model)
        host = mj.decode_plan(
            p,
            lens,
            sm_count=used.sm_count,
            ctas_per_sm=used.ctas_per_sm,
            n_q_tiles=used.n_q_tiles,
            force_splits=force,
            min_chunk_tiles=used.min_chunk_tiles,
            pad_to=pad_to,
        )
        assert status == 0, trial
        assert chunk == host.chunk_tiles, trial
        assert np.array_equal(ns, host.n_splits), trial
        assert np.array_equal(work, host.work), trial
        ref = plan_ref(lens.tolist(), h_k, used.n_q_tiles, 152, used.ctas_per_sm, ms, force, used.min_chunk_tiles, pad_to)
        assert [tuple(x) for x in work.tolist()] == [tuple(x) for x in ref.work], trial


def test_status_word():
    p = mj.make_params(4, 1, 8, 4, 16, 64, 4 * 64, True, mj.MJ_BF16, 16, 128, 0, 0)
    # a length past max_blocks * page_size
    *_, status = device_plan(p, [100, 2000, 64 * 16 + 1, 5], 64)
    assert status == mj.MJ_ERR_INVALID_ARG
    # more items than pad_to
    *_, status = device_plan(p, [1000, 1000, 1000, 1000], 2, ctas_per_sm=24)
    assert status == mj.MJ_ERR_CAPACITY
    # force_splits above max_splits: the chunk floor ceil(T / max_splits) holds
    p1 = mj.make_params(2, 1, 8, 4, 16, 512, 2 * 512, True, mj.MJ_BF16, 2, 128, 0, 0)
    _, work, ns, chunk, status = device_plan(p1, [8000, 8000], 64, force_splits=5)
    assert status == 0 and chunk == 32 and ns.tolist() == [2, 2]


def _decode(s, work, max_n_splits, stream=None):
    mj.decode_attn(
        s.params,
        q=s.q_packed,
        k_cache=s.k_cache,
        v_cache=s.v_cache,
        block_table=s.block_table,
        seq_lens=s.seq_lens,
        work=work,
        n_splits=s.n_splits,
        q_descale=s.q_descale,
        k_descale=s.k_descale,
        v_descale=s.v_descale,
        o=s.o_packed,
        lse=s.lse,
        workspace=s.workspace,
        softmax_scale=s.w.softmax_scale,
        scale_o=s.w.scale_o,
        max_n_splits=max_n_splits,
        stream=stream,
    )


@pytest.mark.parametrize(
    "cfg,kw,kernel",
    [
        (2, dict(num_seqs=6, len_range=(1500, 4000)), 0),  # swap-AB, splits
        (4, dict(num_seqs=3, len_range=(1000, 3000)), 0),  # query rows
        (3, dict(num_seqs=3, len_range=(6000, 300), max_splits=64), 0),  # fully-fp8, many splits
    ],
)
def test_graph_of_device_plan_and_decode_follows_changing_lengths(cfg, kw, kernel):
    w = syn.config(cfg, **kw)
    s = DecodeSession(w, kernel=kernel)
    s.step()  # packs Q (q_len > 1) into the buffer the graph's decode reads
    torch.cuda.synchronize()
    pad_to = mj.decode_plan_max_items(s.params, sm_count=s.sm_count)
    work = torch.zeros((pad_to, 4), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    opts = dict(sm_count=s.sm_count)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        mj.decode_plan_device(s.params, s.seq_lens, work, s.n_splits, pad_to, stream=stream, **opts)
        _decode(s, work, w.max_splits, stream=stream)
    rng = np.random.default_rng(cfg)
    for rep in range(3):
        lens = (w.seq_lens * rng.uniform(0.2, 1.0, w.num_seqs)).astype(np.int32)
        lens[rep % w.num_seqs] = w.seq_lens[rep % w.num_seqs]  # one at full length
        s.seq_lens.copy_(torch.from_numpy(lens))
        s.o_packed.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        w2 = dataclasses.replace(w, seq_lens=lens)
        compare(w2, s.o_host(), s.lse_host())
