"""The seeded input recipe (CPU): the routing and decode token counts, and the small
parity configuration, are the ones the design documents state -- a changed seed, generator
or distribution shows up here before it silently changes a measured workload."""
import torch

import workloads


def test_prefill_routing_counts():
    c = workloads.zipf_routing_counts()
    assert c.dtype == torch.int64 and c.numel() == workloads.N_EXPERTS
    assert int(c.sum()) == 16384 * workloads.TOP_K == 131072     # every token routed to 8 experts
    assert int((c > 0).sum()) == 213 and int(c.max()) == 15900
    assert int(c[0]) == int(c.max())                             # the Zipf bias favours expert 0
    assert torch.equal(c, workloads.zipf_routing_counts())       # seeded


def test_decode_counts():
    c = workloads.moe_decode_counts()
    assert c.numel() == workloads.N_EXPERTS
    assert int(c.min()) >= 1 and int(c.max()) <= 256             # 1..256 tokens per expert
    assert int(c.sum()) == 34495
    assert torch.equal(c, workloads.moe_decode_counts())


def test_offsets_are_the_exclusive_prefix_sum():
    c = torch.tensor([3, 0, 5, 1], dtype=torch.int64)
    assert workloads.offsets_from_counts(c).tolist() == [0, 3, 3, 8, 9]


def test_tiny_config():
    d = workloads.tiny_fprop()
    A, W = d["A"], d["W"]
    assert A.shape == (256, 512) and W.shape == (256, 512)
    assert A.dtype == W.dtype == torch.bfloat16
    # 1% of the 512 columns (5) carry outliers x50: their spread stands far above the rest
    col_max = A.float().abs().amax(0)
    assert int((col_max > 20).sum()) == 5
    assert abs(float(W.float().std()) - 0.02) < 0.002
    assert torch.equal(A, workloads.tiny_fprop()["A"])
