"""GPU parity of the fused fp8 query quantisation + pack (mj_quantize_pack_q)
against the oracle's restatement (oracle/quant_ref.py): codes and descales
bit-exact (the decision of each code is an fp32 division and a round to
nearest even on both sides), then the decode on those codes against the
fp64 attention oracle."""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle.layout_ref import unpack_o_ref
from oracle.quant_ref import quantize_pack_q_ref
from paged_fp8_kv_gb300 import quantize_pack_q
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


def bf16_values(rng, shape, scale=1.0, kind="normal"):
    """float32 values exactly representable in bf16 (the kernel's input)."""
    if kind == "normal":
        x = rng.normal(0, scale, shape)
    elif kind == "wide":  # magnitudes over many binades: subnormal codes after scaling
        x = rng.normal(0, 1, shape) * np.exp2(rng.integers(-20, 4, shape))
    else:
        raise ValueError(kind)
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()


def run_kernel(qf, num_seqs, q_len, h_k, h_r):
    d = qf.shape[-1]
    q = torch.from_numpy(qf).to(torch.bfloat16).cuda()
    q8 = torch.full((num_seqs, h_k, q_len * h_r, d), 0xAB, dtype=torch.uint8, device="cuda")
    ds = torch.full((num_seqs, h_k), float("nan"), dtype=torch.float32, device="cuda")
    quantize_pack_q(q, q8, ds, num_seqs, q_len, h_k, h_r)
    torch.cuda.synchronize()
    return q8.cpu().numpy(), ds.cpu().numpy()


@pytest.mark.parametrize(
    "num_seqs,q_len,h_k,h_r,d,kind,scale",
    [
        (8, 1, 1, 16, 128, "normal", 1.0),  # fully-fp8 skewed shape
        (4, 4, 8, 8, 128, "normal", 3.0),  # spec-verify shape
        (3, 5, 3, 5, 128, "normal", 0.01),  # ragged heads and tokens
        (2, 2, 2, 4, 64, "wide", 1.0),  # subnormal and zero codes
        (2, 16, 1, 32, 128, "normal", 1.0),  # 512 rows per group (two passes over a 128 KB group)
        (5, 1, 2, 3, 16, "normal", 100.0),  # smallest head_dim
    ],
)
def test_codes_and_descales_bit_exact(num_seqs, q_len, h_k, h_r, d, kind, scale):
    rng = np.random.default_rng(num_seqs * 1000 + q_len * 10 + h_r)
    qf = bf16_values(rng, (num_seqs * q_len, h_k * h_r, d), scale, kind)
    qf[:q_len, :h_r] = 0.0  # an all-zero group: descale 1e-6 / 448, every code 0
    codes, ds = run_kernel(qf, num_seqs, q_len, h_k, h_r)
    ref_codes, ref_ds = quantize_pack_q_ref(qf, num_seqs, q_len, h_k, h_r)
    assert np.array_equal(ds.view(np.uint32), ref_ds.view(np.uint32))
    assert np.array_equal(codes, ref_codes)


def test_decode_on_quantised_q_matches_oracle():
    # bf16 Q -> fused quantisation on the GPU -> fully-fp8 decode, against
    # the fp64 oracle on the oracle's own quantisation of the same Q
    w = syn.config(3, num_seqs=4, len_range=(3000, 300), max_splits=16)
    rng = np.random.default_rng(97)
    qf = bf16_values(rng, (w.num_seqs * w.q_len, w.h_q, w.head_dim))
    ref_codes, ref_ds = quantize_pack_q_ref(qf, w.num_seqs, w.q_len, w.h_k, w.h_r)
    w2 = dataclasses.replace(
        w,
        q=np.ascontiguousarray(unpack_o_ref(ref_codes, w.num_seqs, w.q_len, w.h_k, w.h_r)),
        q_descale=np.ascontiguousarray(ref_ds),
    )
    s = DecodeSession(w2)
    s.q_packed.fill_(0)
    s.q_descale.fill_(float("nan"))
    q = torch.from_numpy(qf).to(torch.bfloat16).cuda()
    quantize_pack_q(q, s.q_packed, s.q_descale, w.num_seqs, w.q_len, w.h_k, w.h_r)
    s.decode()
    torch.cuda.synchronize()
    assert np.array_equal(s.q_packed.cpu().numpy().reshape(ref_codes.shape), ref_codes)
    compare(w2, s.o_host(), s.lse_host())


def test_graph_capture_and_determinism():
    rng = np.random.default_rng(3)
    qf = bf16_values(rng, (4 * 2, 8 * 4, 128))
    q = torch.from_numpy(qf).to(torch.bfloat16).cuda()
    q8 = torch.empty((4, 8, 8, 128), dtype=torch.uint8, device="cuda")
    ds = torch.empty((4, 8), dtype=torch.float32, device="cuda")
    quantize_pack_q(q, q8, ds, 4, 2, 8, 4)
    torch.cuda.synchronize()
    a8, ads = q8.clone(), ds.clone()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    q8.zero_()
    with torch.cuda.graph(g, stream=stream):
        quantize_pack_q(q, q8, ds, 4, 2, 8, 4, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a8, q8) and torch.equal(ads, ds)
