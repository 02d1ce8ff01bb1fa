"""Host-side pieces the extend measurements rest on (CPU only): the FLOP count
of the bench row, the seeded E4M3 code generator and the extend input layout."""
import numpy as np
import torch

import workloads
from bench import extend_flops


def test_extend_flops_is_the_count_of_visible_pairs():
    """4 d flops per (chunk token, query head, visible key); token t of a
    chunk with prefix P sees P + t + 1 keys -- counted here pair by pair."""
    e = workloads.extend_custom((0, 5, 37), (3, 1, 20), 8, 2)
    pairs = 0
    for P, C in zip(e.prefix_lens, e.chunk_lens):
        for t in range(C):
            pairs += sum(1 for _ in range(P + t + 1))
    assert extend_flops(e) == 4 * 128 * 8 * pairs


def test_e4m3_codes_are_finite_and_in_range():
    gen = torch.Generator().manual_seed(3)
    codes = workloads.e4m3_codes((200000,), gen)
    assert codes.dtype == torch.uint8
    assert not ((codes & 0x7F) == 0x7F).any()                # no NaN code
    vals = codes.view(torch.float8_e4m3fn).float()
    mag = vals.abs()
    assert mag.max() <= 3.75 and mag[mag > 0].min() >= 2.0 ** -6
    zeros = (mag == 0).float().mean().item()
    assert 0.02 < zeros < 0.045                                # about 1 in 32
    assert 0.45 < (vals < 0).float().mean().item() < 0.55


def test_extend_input_layout():
    e = workloads.extend_make("ext_small")
    x = workloads.extend_inputs(e)
    qi, ki, pl = x["q_indptr"].numpy(), x["kv_indptr"].numpy(), x["prefix_lens"].numpy()
    np.testing.assert_array_equal(np.diff(qi), e.chunk_lens)
    assert qi[0] == 0 and qi[-1] == e.q_rows == x["q"].shape[0]
    # sequences sit in the workspace in order, EXTEND_GAP unused rows before each
    ends = ki + pl
    assert ki[0] == workloads.EXTEND_GAP
    np.testing.assert_array_equal(ki[1:] - ends[:-1], workloads.EXTEND_GAP)
    assert ends.max() <= e.prefix_rows == x["k_prefix"].shape[0]
    assert x["q"].dtype == torch.bfloat16 and x["k_chunk"].shape == (e.q_rows, e.num_kv_heads, 128)
    # the same seed gives the same inputs
    y = workloads.extend_inputs(e)
    assert torch.equal(x["k_prefix"], y["k_prefix"]) and torch.equal(x["q"], y["q"])
