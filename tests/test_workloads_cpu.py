"""The seeded input generators (CPU): shapes, types, value ranges and
determinism of the workloads the benchmark and the full-size tests use, at
reduced sizes where the generator takes them."""

import numpy as np
import torch

import oracle
import workloads


def test_generators_are_seeded():
    a = workloads.grouped_qweights(device="cpu", M=64, K=128, N=32, G=4, bits=8)
    b = workloads.grouped_qweights(device="cpu", M=64, K=128, N=32, G=4, bits=8)
    for k in ("input", "weights_q", "w_scale", "w_zero_point", "bias", "group_indices"):
        assert torch.equal(a[k], b[k]), k


def test_int8_experts():
    d = workloads.grouped_qweights(device="cpu", M=64, K=128, N=32, G=4, block=64)
    assert d["weights_q"].dtype == torch.int8 and tuple(d["weights_q"].shape) == (4, 128, 32)
    assert tuple(d["w_scale"].shape) == (4, 2, 32) and d["w_scale"].dtype == torch.bfloat16
    assert d["w_zero_point"].dtype == torch.int8 and int(d["w_zero_point"].abs().max()) <= 8
    assert "packed4" not in d


def test_int4_experts_packed_two_per_byte():
    d = workloads.grouped_qweights(device="cpu", M=64, K=128, N=32, G=4, bits=4)
    assert d["packed4"] == "int4"
    assert d["weights_q"].dtype == torch.uint8 and tuple(d["weights_q"].shape) == (4, 128, 16)
    assert d["w_zero_point"].dtype == torch.uint8 and tuple(d["w_zero_point"].shape) == (4, 1, 16)
    q = oracle.unpack_4bit(d["weights_q"].numpy(), True)
    z = oracle.unpack_4bit(d["w_zero_point"].numpy(), True)
    assert q.shape == (4, 128, 32) and q.min() >= -8 and q.max() <= 7
    assert set(np.unique(z).tolist()) <= {-1, 0, 1}
    # uniform random bytes: every int4 value occurs
    assert set(np.unique(q).tolist()) == set(range(-8, 8))
    s = d["w_scale"].float()
    assert float(s.min()) >= 2.39e-3 and float(s.max()) <= 4.31e-3


def test_group_indices_two_distinct_groups_per_token():
    d = workloads.grouped_bf16(device="cpu", M=256, K=64, N=32, G=8)
    gi = d["group_indices"]
    assert tuple(gi.shape) == (256, 2) and gi.dtype == torch.int32
    assert bool((gi[:, 0] != gi[:, 1]).all()) and int(gi.min()) >= 0 and int(gi.max()) < 8
