"""The five workloads end to end on the GPU (build -> kernel map -> conv).

Reduced sizes: bit-exact topology and kernel maps against the CPU oracle, conv
against the oracle within tolerance.  Full sizes (the sizes the benchmark
times): topology bit-exact against an independent numpy derivation from the
sorted unique keys, kernel maps bit-exact on every output and slot (numpy
searchsorted in the sorted keys), conv within tolerance on sampled output rows
recomputed in numpy fp64.
"""
import numpy as np
import pytest

import oracle
from sparse_convolution_gb300 import synth
from tests import gpu_common as G
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _oracle_parity(w, conv_rows=None):
    """Build + kmap (+ conv) vs the oracle; conv on all rows unless conv_rows."""
    import sparse_convolution_gb300 as fvx

    coords, offs = w["coords"], w["batch_offsets"]
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    G.assert_topology_equal(g, og)
    x = None
    for i, cv in enumerate(w["convs"]):
        stride = cv["stride"]
        gout = g if stride == 1 else g.coarsen(2)
        ogout = og if stride == 1 else og.coarsen(2)
        if stride != 1:
            G.assert_topology_equal(gout, ogout)
        km = fvx.KernelMap(g, gout, stride)
        okm = oracle.KernelMap(og, ogout, stride)
        G.assert_kmap_equal(km, okm)
        if x is None:
            if w["dtype"] == "f32":
                import torch

                x = torch.from_numpy(synth.features(w["seed"] + 10, g.n_active, cv["cin"], w["feat_kind"])).cuda()
            else:
                x, _ = G.bf16_inputs(w["seed"] + 10, g.n_active, cv["cin"], cv["cout"], w["feat_kind"])
        import torch

        W = torch.from_numpy(synth.weights(w["seed"] + 20 + i, cv["cin"], cv["cout"])).cuda()
        W = W if w["dtype"] == "f32" else W.bfloat16()
        y = fvx.sparse_conv(g, gout, km, x, W)
        kern = fvx.last_conv_kernel()
        fvx.device_status()
        tol = G.F32_TOL if w["dtype"] == "f32" else G.BF16_TOL
        if conv_rows is None:
            yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
            G.assert_conv_close(G.np_(y.float()), yo, ao, tol)
        else:
            rows = np.random.default_rng(i).choice(gout.n_active, size=min(conv_rows, gout.n_active), replace=False)
            yo, ao = oracle.conv_rows(og, ogout, stride, rows, G.as_f64(x), G.as_f64(W))
            G.assert_conv_close(G.np_(y.float())[rows], yo, ao, tol)
        if w["dtype"] != "f32":
            # the next conv reads this one's bf16-rounded output (LiDAR: subm 128 -> stride-2 128->256)
            yb = fvx.sparse_conv(g, gout, km, x, W, out_dtype=torch.bfloat16)
            if fvx.last_conv_kernel() == kern:
                assert torch.equal(yb, y.bfloat16())
            else:  # wider inputs: fp32 output by the halo passes, bf16 output by the pair lists
                sel = np.arange(gout.n_active) if conv_rows is None else rows
                G.assert_conv_close(G.np_(yb.float())[sel], yo, ao, tol)
            y = yb
        x = y
        if stride != 1:
            break


def test_tiny_shell_full_oracle(cuda_device):
    _oracle_parity(synth.tiny_shell())


def test_leaf_dense_reduced_oracle(cuda_device):
    _oracle_parity(synth.leaf_dense(scale=0.3))


def test_narrow_band_reduced_oracle(cuda_device):
    _oracle_parity(synth.narrow_band(scale=0.125))


def test_lidar_full_oracle(cuda_device):
    _oracle_parity(synth.lidar(), conv_rows=3000)


def test_batched_reduced_oracle(cuda_device):
    _oracle_parity(synth.batched_narrow_band(scale=0.125))


# ---------------------------------------------------------------- full sizes

def _full_size(w, n_conv_rows=3000):
    import torch

    import sparse_convolution_gb300 as fvx

    coords, offs = w["coords"], w["batch_offsets"]
    g = G.gpu_grid(coords, offs)
    uniq, ijk, vb = G.check_build_full(g, coords, offs)
    rng = np.random.default_rng(99)
    x = None
    for i, cv in enumerate(w["convs"]):
        stride = cv["stride"]
        if stride == 1:
            gout, uniq_out, ijk_out, vb_out = g, uniq, ijk, vb
        else:
            gout = g.coarsen(2)
            exp = np.unique(H.key64(vb, np.floor_divide(ijk, 2)))
            t = {k: G.np_(v) for k, v in gout.topology().items()}
            vb_out = np.repeat(np.arange(len(offs) - 1), np.diff(t["voxel_batch_offsets"]))
            assert np.array_equal(H.key64(vb_out, t["ijk"]), exp)
            ijk_out = t["ijk"]
        km = fvx.KernelMap(g, gout, stride)
        G.check_kmap_full(km, uniq, ijk_out, vb_out, stride)
        if x is None:
            if w["dtype"] == "f32":
                x = torch.from_numpy(synth.features(w["seed"] + 10, g.n_active, cv["cin"], w["feat_kind"])).cuda()
            else:
                x, _ = G.bf16_inputs(w["seed"] + 10, g.n_active, cv["cin"], cv["cout"], w["feat_kind"])
        W = torch.from_numpy(synth.weights(w["seed"] + 20 + i, cv["cin"], cv["cout"])).cuda()
        W = W if w["dtype"] == "f32" else W.bfloat16()
        y = fvx.sparse_conv(g, gout, km, x, W)
        fvx.device_status()
        crow = np.sort(rng.choice(gout.n_active, size=min(n_conv_rows, gout.n_active), replace=False))
        nbr = G.neighbours_independent(uniq, ijk_out, vb_out, stride, crow)
        yr, ar = G.conv_rows_independent(nbr, G.as_f64(x), G.as_f64(W))
        tol = G.F32_TOL if w["dtype"] == "f32" else G.BF16_TOL
        G.assert_conv_close(G.np_(y.float())[crow], yr, ar, tol)
        if w["dtype"] != "f32":
            y = fvx.sparse_conv(g, gout, km, x, W, out_dtype=torch.bfloat16)
        x = y
        if stride != 1:
            break


def test_leaf_dense_full_size(cuda_device):
    _full_size(synth.leaf_dense())


def test_narrow_band_full_size(cuda_device):
    _full_size(synth.narrow_band())


def test_lidar_full_size(cuda_device):
    _full_size(synth.lidar())


def test_batched_full_size(cuda_device):
    _full_size(synth.batched_narrow_band())
