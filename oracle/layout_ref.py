"""Plain numpy restatement of the query/output row permutation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: the "mjolnir/t5_decode.py" page, `pack_q` / `unpack_o` and the module
docstring: packed row n of kv head g is query token qi = n // h_r of query
head g*h_r + n % h_r, i.e. (b, q_len, h_k, h_r, d) -> (b, h_k, q_len, h_r, d).
"""

import numpy as np


def pack_q_ref(q_vllm: np.ndarray, num_seqs: int, q_len: int, h_k: int, h_r: int) -> np.ndarray:
    d = q_vllm.shape[-1]
    return (
        q_vllm.reshape(num_seqs, q_len, h_k, h_r, d).transpose(0, 2, 1, 3, 4).reshape(num_seqs, h_k, q_len * h_r, d)
    )


def unpack_o_ref(o_packed: np.ndarray, num_seqs: int, q_len: int, h_k: int, h_r: int) -> np.ndarray:
    d = o_packed.shape[-1]
    return (
        o_packed.reshape(num_seqs, h_k, q_len, h_r, d).transpose(0, 2, 1, 3, 4).reshape(num_seqs * q_len, h_k * h_r, d)
    )
