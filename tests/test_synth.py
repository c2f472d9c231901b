"""The seeded input generators (host only): shapes, types, determinism and
the cluster structure each workload states."""
import torch

from mixture_top_attention_mita_b300 import synth


def test_deterministic_and_typed():
    w = synth.WORKLOADS["deit_s"].scaled(B=2, H=2)
    a, b = synth.make_inputs(w), synth.make_inputs(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.bfloat16 and x.shape == (2, 2, 196, 64)


def test_hires56_clusters_straddle_the_pooling_bins():
    # Cluster ids are fixed per 8 x 8 tile of the 56 x 56 grid, the tiles
    # offset by 4 tokens from the 8 x 8 pooling bins: contiguous, not aligned.
    w = synth.WORKLOADS["hires56"].scaled(B=1, H=2)
    assert w.patch == 8 and w.patch_offset == 4
    *_, ids = synth.make_inputs(w, return_ids=True)
    g = ids.reshape(2, 56, 56)
    for y0 in range(-4, 56, 8):
        for x0 in range(-4, 56, 8):
            tile = g[:, max(0, y0):y0 + 8, max(0, x0):x0 + 8]
            assert (tile == tile[:, :1, :1]).all()          # one id per offset tile
    mixed = 0
    for r in range(7):
        for c in range(7):
            mixed += int(g[0, 8 * r:8 * r + 8, 8 * c:8 * c + 8].unique().numel() > 1)
    assert mixed >= 30    # most pooling bins see two to four clusters


def test_cluster_patch_without_offset_aligns_with_bins():
    w = synth.WORKLOADS["hires56"].scaled(B=1, H=1, patch_offset=0)
    *_, ids = synth.make_inputs(w, return_ids=True)
    g = ids.reshape(56, 56)
    for r in range(7):
        for c in range(7):
            assert g[8 * r:8 * r + 8, 8 * c:8 * c + 8].unique().numel() == 1
