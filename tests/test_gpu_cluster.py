"""GPU parity of the online V clustering (fp8attn_v_cluster) against the oracle:
the permutation and the cluster ids are integer results and must match
exactly, on small cases that span several 1024-token chunks with a ragged
tail, on the degenerate cases, and on sampled heads of the full Wan2.2-shaped
workload (B=1, H=40, T=75600) in the configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import bit_attention_video_e4m3_gb300 as fa
from bit_attention_video_e4m3_gb300.workloads import bf16_bits, make_workload
from oracle import cluster as OC
from oracle.bf16 import bf16_from_bits
from tests import parity as P

pytestmark = pytest.mark.gpu


def _check_head(w, perm, labels, b, h, K, r, iters):
    v = bf16_from_bits(bf16_bits(w.v[b, :, h, :]))
    ref_perm, ref_labels = OC.cluster_head(v, n_clusters=K, n_dims=r, iters=iters)
    got_labels = labels[b, h].cpu().numpy()
    assert np.array_equal(got_labels, ref_labels), (b, h, np.flatnonzero(got_labels != ref_labels)[:10])
    assert np.array_equal(perm[b, h].cpu().numpy(), ref_perm), (b, h)


@pytest.mark.parametrize("name,B,H,T,K,r,iters", [
    ("tiny", 1, 2, 1024, 32, 8, 4),          # defaults, one full chunk
    ("wan22", 1, 3, 2500, 16, 8, 3),         # clustered V with outliers, ragged third chunk
    ("wan22", 1, 2, 3333, 64, 12, 2),        # 16-wide code rows, the largest K
    ("tiny", 1, 2, 777, 7, 16, 0),           # assignment to the seeds only
    ("tiny", 1, 1, 5, 8, 3, 2),              # fewer tokens than clusters
    ("tiny", 1, 1, 1, 4, 8, 4),              # a single token
])
def test_cluster_parity(name, B, H, T, K, r, iters):
    w = make_workload(name, device="cuda", T=T, H=H, seed=11)
    perm, labels = fa.v_cluster(w.v, n_clusters=K, n_dims=r, iters=iters, with_labels=True)
    torch.cuda.synchronize()
    for h in range(H):
        _check_head(w, perm, labels, 0, h, K, r, iters)


def test_cluster_parity_batched():
    # two batch entries with different data: the (batch, head) pairs must not mix
    w = make_workload("wan22", device="cuda", T=1500, H=2, seed=12)
    w2 = make_workload("wan22", device="cuda", T=1500, H=2, seed=13)
    w.v = torch.cat([w.v, w2.v], dim=0).contiguous()
    w.B = 2
    perm, labels = fa.v_cluster(w.v, n_clusters=24, n_dims=8, iters=3, with_labels=True)
    for b in range(2):
        for h in range(2):
            _check_head(w, perm, labels, b, h, 24, 8, 3)


def test_degenerate_inputs_give_the_identity():
    for fill in (0.0, 2.5):
        v = torch.full((1, 300, 2, 128), fill, dtype=torch.bfloat16, device="cuda")
        perm, labels = fa.v_cluster(v, n_clusters=16, with_labels=True)
        ident = torch.arange(300, dtype=torch.int32, device="cuda").expand(1, 2, 300)
        assert torch.equal(perm, ident) and torch.all(labels == 0)
    w = make_workload("tiny", device="cuda", T=900, H=1, seed=14)
    perm = fa.v_cluster(w.v, n_clusters=1)
    assert torch.equal(perm[0, 0].cpu(), torch.arange(900, dtype=torch.int32))


def test_full_size_wan22_sampled_heads():
    w = make_workload("wan22", device="cuda")
    perm, labels = fa.v_cluster(w.v, with_labels=True)       # defaults: K=32, r=8, 4 rounds
    torch.cuda.synchronize()
    # every head: a permutation that sorts the cluster ids stably
    T = w.T
    srt, _ = torch.sort(perm.long(), dim=-1)
    assert torch.equal(srt, torch.arange(T, device="cuda").expand_as(srt))
    lab_sorted = torch.gather(labels, 2, perm.long())
    assert torch.all(lab_sorted[..., 1:] >= lab_sorted[..., :-1])
    same = lab_sorted[..., 1:] == lab_sorted[..., :-1]
    assert torch.all(~same | (perm[..., 1:] > perm[..., :-1]))
    for h in (0, 17, 39):
        _check_head(w, perm, labels, 0, h, 32, 8, 4)


def test_clustered_order_feeds_the_prep():
    # the clustering permutation goes straight into the prep's V gather: the prep
    # result must equal the oracle's prep under the oracle's permutation
    w = make_workload("wan22", device="cuda", T=4000, H=2, seed=15)
    w.perm = fa.v_cluster(w.v)
    pp = fa.prep(w.q, w.k, w.v, perm=w.perm, vsmooth=True)
    for h in range(w.H):
        _, _, v, _ = P.head_arrays(w, 0, h)
        ref_perm, _ = OC.cluster_head(v)
        assert np.array_equal(w.perm[0, h].cpu().numpy(), ref_perm)
        ref = P.oracle_prep_head(w, 0, h)
        P.assert_prep_bitexact(pp, ref, 0, h)
