"""GPU parity at full size through the library's automatic kernel choice
(MJ_KERNEL_AUTO), the launch configuration the benchmark times.

For every workload of the benchmark's configurations (and the sweep points
whose packed-row count picks a different kernel instance) the whole batch
runs at its full size and sampled (sequence, kv head) units, always
including the longest sequence and the last kv head, are compared with the
fp64 oracle element by element.  Each case also asserts which kernel the
library chose, so that a change of the automatic choice cannot leave a
kernel instance untested at full size.
"""

import numpy as np
import pytest
import torch

from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare, sample_units

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


CASES = [
    # (config, workload options, kernel the library picks)
    (2, {}, "tc_r8_bf16"),
    (3, {}, "tc_r16_e4m3"),
    (4, {}, "qm_r32_bf16"),
    (4, {"variant": "noncausal"}, "qm_r64_bf16"),
    (5, {"h_r": 16, "q_len": 1}, "tc_r16_bf16"),
    (5, {"h_r": 32, "q_len": 1}, "qm_r32_bf16"),
    (5, {"h_r": 16, "q_len": 2}, "qm_r32_bf16"),
    (5, {"h_r": 16, "q_len": 4}, "qm_r64_bf16"),
    (5, {"h_r": 32, "q_len": 4}, "qm_bf16"),
    (5, {"h_r": 16, "q_len": 16}, "qm_pair_bf16"),
    (5, {"h_r": 32, "q_len": 16}, "qm_pair_bf16"),
]


@pytest.mark.parametrize("cfg,opts,kernel", CASES, ids=[f"cfg{c}-{k}-{'-'.join(f'{a}{b}' for a, b in o.items())}" for c, o, k in CASES])
def test_full_size_automatic_kernel(cfg, opts, kernel):
    w = syn.config(cfg, **opts)
    s = DecodeSession(w)  # MJ_KERNEL_AUTO
    assert s.kernel == kernel
    s.fill_workspace(float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s.step(status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    longest = int(np.argmax(w.seq_lens))
    units = sample_units(w, 8, seed=cfg, include=[(longest, w.h_k - 1), (longest, 0), (w.num_seqs - 1, w.h_k - 1)])
    compare(w, s.o_host(), s.lse_host(), units=units)
