"""Host checks of the seeded input generator (no GPU, no method arithmetic)."""
import math

import numpy as np
import torch

import workloads as wl
from oracle import qkv_cte_oracle as O


def test_deterministic_and_valid_codes():
    call = wl.workload("tiny")[0]
    a = wl.make_inputs(call)
    b = wl.make_inputs(call)
    for k in a:
        if a[k] is None:
            assert b[k] is None
        else:
            assert torch.equal(a[k], b[k]), k
    for k in ("A", "W"):
        codes = a[k].numpy()
        assert not np.any((codes & 0x7F) == 0x7F), "NaN code generated"
    sf = a["w_sf"].numpy()
    assert sf.min() >= 1 and sf.max() <= 254
    assert a["A"].shape == (256, 512) and a["W"].shape == (1536, 512)
    assert a["w_sf"].shape == (1536, 16)


def test_row_quantiser_recipe():
    """Every row's largest code is +-448 and the scale is amax/448."""
    call = wl.custom_call(tokens=64, hidden=256, n_q_heads=1, n_kv_heads=1, d_head=16, seed=3)
    inp = wl.make_inputs(call)
    dec = O.decode_e4m3(inp["A"].numpy())
    assert np.all(np.max(np.abs(dec), axis=1) == 448.0)
    assert np.all(inp["a_scale"].numpy() > 0)


def test_mx_quantiser_recipe():
    """No block clips and the block maximum lands in (224, 448]."""
    call = wl.custom_call(tokens=8, hidden=256, n_q_heads=2, n_kv_heads=1, d_head=16, seed=4)
    inp = wl.make_inputs(call)
    dec = O.decode_e4m3(inp["W"].numpy()).reshape(64, 8, 32)
    amax = np.max(np.abs(dec), axis=2)
    assert np.all(amax <= 448.0) and np.all(amax > 224.0 / 1.2)


def test_rope_tables_rotate_half_structure():
    call = wl.workload("short")[0]
    cos, sin = wl.rope_tables(call, 300)
    assert cos.shape == (300, 128)
    assert torch.equal(cos[:, :64], cos[:, 64:]) and torch.equal(sin[:, :64], sin[:, 64:])
    # token 0 sits at the grid origin: zero angle everywhere
    assert torch.all(cos[0] == 1) and torch.all(sin[0] == 0)
    # token 1 is (f=0, h=0, w=1): only the w pairs (the last 21) rotate
    ang = wl.rope_positions(call, 2)[1]
    assert torch.all(ang[:43] == 0) and torch.all(ang[43:] != 0)
    assert math.isclose(float(ang[43]), 1.0)


def test_outlier_rows():
    call = wl.custom_call(tokens=2000, hidden=128, n_q_heads=1, n_kv_heads=1, d_head=16,
                          outlier_frac=0.001, seed=9)
    inp = wl.make_inputs(call)
    scale = inp["a_scale"].numpy()
    big = np.sort(scale)[-2:]
    assert big.min() > 5 * np.median(scale)


def test_sample_rows():
    call = wl.workload("wan480p")[0]
    r = wl.sample_rows(call, 4096)
    assert len(r) == 4096 and int(r[-1]) == call.tokens - 1
    assert len(torch.unique(r)) == 4096
