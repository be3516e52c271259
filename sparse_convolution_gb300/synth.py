"""Seeded synthetic workloads for the sparse-voxel hot path.

These generators produce INPUTS only (voxel coordinates, CSR batch offsets,
features and weights).  They hold none of the method's arithmetic: no tree,
no index order, no neighbour search, no convolution.  Both the CUDA path and
the CPU oracle are fed from here.

The geometries stand in for the datasets the pages measure on (SemanticKITTI,
nuScenes, KartonCity, Waymo), which are not available; see each function.
Every generator uses ``numpy.random.default_rng(seed)`` and shuffles rows with
the same generator.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# geometry helpers (pure input construction)
# ---------------------------------------------------------------------------


def _finish(coords_list, rng, dup_frac=0.0):
    """Concatenate per-batch unique voxel sets, add duplicate rows, shuffle.

    Returns dict(coords int32 [N,3], batch_offsets int64 [B+1], n_unique [B]).
    ``dup_frac`` is the fraction of the FINAL rows of each batch that repeat a
    uniformly chosen row of that batch's unique set.
    """
    rows, offs, nu = [], [0], []
    for c in coords_list:
        c = np.asarray(c, dtype=np.int32).reshape(-1, 3)
        u = c.shape[0]
        nu.append(u)
        if dup_frac > 0 and u > 0:
            n_total = int(round(u / (1.0 - dup_frac)))
            extra = c[rng.integers(0, u, size=n_total - u)]
            c = np.concatenate([c, extra], axis=0)
        c = c[rng.permutation(c.shape[0])]
        rows.append(c)
        offs.append(offs[-1] + c.shape[0])
    coords = np.concatenate(rows, axis=0) if rows else np.zeros((0, 3), np.int32)
    return dict(coords=np.ascontiguousarray(coords, dtype=np.int32),
                batch_offsets=np.asarray(offs, dtype=np.int64),
                n_unique=np.asarray(nu, dtype=np.int64))


def _grid_centres(lo, hi):
    return np.arange(lo, hi, dtype=np.float64) + 0.5


def shell_voxels(box=64, radius=24.0, half_width=2.0):
    """Voxels whose centre lies within ``half_width`` of a sphere of ``radius``
    centred in a ``box``^3 cube."""
    c = _grid_centres(0, box) - box / 2.0
    X, Y, Z = np.meshgrid(c, c, c, indexing="ij")
    r = np.sqrt(X * X + Y * Y + Z * Z)
    sel = np.abs(r - radius) <= half_width
    return np.stack(np.nonzero(sel), axis=1).astype(np.int32)


def ellipsoid_voxels(rng, box=256, n=40, rmin=8.0, rmax=40.0):
    """Union of ``n`` solid axis-aligned ellipsoids, centres uniform in the box,
    per-axis radii uniform in [rmin, rmax]; clipped to the box."""
    occ = np.zeros((box, box, box), dtype=bool)
    c1 = _grid_centres(0, box)
    for _ in range(n):
        ctr = rng.uniform(0, box, size=3)
        rad = rng.uniform(rmin, rmax, size=3)
        lo = np.clip(np.floor(ctr - rad).astype(int), 0, box)
        hi = np.clip(np.ceil(ctr + rad).astype(int) + 1, 0, box)
        xs = (c1[lo[0]:hi[0]] - ctr[0]) / rad[0]
        ys = (c1[lo[1]:hi[1]] - ctr[1]) / rad[1]
        zs = (c1[lo[2]:hi[2]] - ctr[2]) / rad[2]
        inside = (xs[:, None, None] ** 2 + ys[None, :, None] ** 2 + zs[None, None, :] ** 2) <= 1.0
        occ[lo[0]:hi[0], lo[1]:hi[1], lo[2]:hi[2]] |= inside
    return np.stack(np.nonzero(occ), axis=1).astype(np.int32)


def _sphere_band(ctr, r, band, box):
    """Voxels (centre p = idx + 0.5) with | |p - ctr| - r | <= band, in the box."""
    ext = r + band + 1.0
    lo = np.clip(np.floor(ctr - ext).astype(np.int64), 0, box)
    hi = np.clip(np.ceil(ctr + ext).astype(np.int64) + 1, 0, box)
    I, J = np.meshgrid(np.arange(lo[0], hi[0]), np.arange(lo[1], hi[1]), indexing="ij")
    I = I.ravel()
    J = J.ravel()
    d2 = (I + 0.5 - ctr[0]) ** 2 + (J + 0.5 - ctr[1]) ** 2
    rout2 = (r + band) ** 2
    rin = max(r - band, 0.0)
    keep = d2 <= rout2
    I, J, d2 = I[keep], J[keep], d2[keep]
    smax = np.sqrt(rout2 - d2)
    smin = np.sqrt(np.maximum(rin * rin - d2, 0.0))
    out = []
    for sign in (-1.0, 1.0):
        # z - ctr in sign*[smin, smax]  with z = k + 0.5
        a = ctr[2] - 0.5 + (np.where(sign < 0, -smax, smin))
        b = ctr[2] - 0.5 + (np.where(sign < 0, -smin, smax))
        k0 = np.maximum(np.ceil(a).astype(np.int64), 0)
        k1 = np.minimum(np.floor(b).astype(np.int64), box - 1)
        # where the two intervals touch (smin == 0) a k may be emitted twice;
        # the union step removes repeats
        cnt = np.maximum(k1 - k0 + 1, 0)
        tot = int(cnt.sum())
        if tot == 0:
            continue
        rep = np.repeat(np.arange(cnt.shape[0]), cnt)
        start = np.repeat(np.cumsum(cnt) - cnt, cnt)
        k = k0[rep] + (np.arange(tot) - start)
        out.append(np.stack([I[rep], J[rep], k], axis=1))
    if not out:
        return np.zeros((0, 3), np.int64)
    v = np.concatenate(out, axis=0)
    # exact re-check of the band condition on the centres
    p = v + 0.5
    d = np.sqrt(((p - ctr) ** 2).sum(axis=1)) - r
    return v[np.abs(d) <= band]


def narrow_band_voxels(rng, box=2048, rmin=20.0, rmax=150.0, band=1.5, min_voxels=None, n_spheres=None,
                       centre_lo=0.0, centre_hi=1.0):
    """Band of half-width ``band`` around the zero level set of a union of
    random spheres (centres uniform in [centre_lo, centre_hi) * box per axis,
    radii uniform in [rmin, rmax]).

    Either a fixed ``n_spheres`` or: add spheres (in seed order) until the band
    holds at least ``min_voxels`` voxels.
    """
    spheres, parts, total = [], [], 0
    while True:
        if n_spheres is not None and len(spheres) >= n_spheres:
            break
        ctr = rng.uniform(centre_lo * box, centre_hi * box, size=3)
        r = float(rng.uniform(rmin, rmax))
        spheres.append((ctr, r))
        v = _sphere_band(ctr, r, band, box)
        parts.append(v)
        total += v.shape[0]
        if n_spheres is None and total >= min_voxels * 1.02:
            vox = _band_union(parts, spheres, band, box)
            if vox.shape[0] >= min_voxels:
                return vox
    return _band_union(parts, spheres, band, box)


def _band_union(parts, spheres, band, box):
    v = np.concatenate(parts, axis=0) if parts else np.zeros((0, 3), np.int64)
    key = (v[:, 0] * box + v[:, 1]) * box + v[:, 2]
    key.sort()
    if key.shape[0]:
        key = key[np.concatenate([[True], key[1:] != key[:-1]])]
    v = np.stack([key // (box * box), (key // box) % box, key % box], axis=1)
    # union SDF = min_s(|p - c_s| - r_s); drop voxels deep inside another
    # sphere.  Rows are sorted by x, so the voxels within a sphere's x extent
    # form one slice.
    p = v + 0.5
    keep = np.ones(v.shape[0], dtype=bool)
    for ctr, r in spheres:
        a = np.searchsorted(p[:, 0], ctr[0] - r, side="left")
        b = np.searchsorted(p[:, 0], ctr[0] + r, side="right")
        if a >= b:
            continue
        ps = p[a:b]
        near = np.all(np.abs(ps - ctr) <= r, axis=1)
        if not near.any():
            continue
        d = np.sqrt(((ps[near] - ctr) ** 2).sum(axis=1)) - r
        keep[a + np.nonzero(near)[0][d < -band]] = False
    return v[keep].astype(np.int32)


def lidar_points(rng, beams=64, azimuths=2048, el_lo=-25.0, el_hi=3.0, height=1.8, n_boxes=60,
                 box_lo=1.0, box_hi=5.0, extent=72.0, keep_out=3.0, returns=5, jitter=0.02):
    """A spinning LiDAR at the origin, ``height`` above a ground plane, with
    ``n_boxes`` axis-aligned boxes resting on the ground.  Each ray keeps its
    nearest hit; each hit gives ``returns`` points whose measured range is
    jittered by N(0, jitter), i.e. each point moves along its own ray (range
    noise, the error a time-of-flight sensor makes)."""
    el = np.deg2rad(np.linspace(el_lo, el_hi, beams))
    az = np.arange(azimuths) * (2.0 * np.pi / azimuths)
    E, A = np.meshgrid(el, az, indexing="ij")
    d = np.stack([np.cos(E) * np.cos(A), np.cos(E) * np.sin(A), np.sin(E)], axis=-1).reshape(-1, 3)
    n = d.shape[0]
    t = np.full(n, np.inf)
    down = d[:, 2] < 0
    t[down] = -height / d[down, 2]
    ground = -height
    for _ in range(n_boxes):
        while True:
            cxy = rng.uniform(-extent, extent, size=2)
            if np.any(np.abs(cxy) > keep_out):
                break
        size = rng.uniform(box_lo, box_hi, size=3)
        bmin = np.array([cxy[0] - size[0] / 2, cxy[1] - size[1] / 2, ground])
        bmax = np.array([cxy[0] + size[0] / 2, cxy[1] + size[1] / 2, ground + size[2]])
        with np.errstate(divide="ignore", invalid="ignore"):
            inv = 1.0 / d
            t0 = bmin * inv
            t1 = bmax * inv
        tmin = np.nanmax(np.minimum(t0, t1), axis=1)
        tmax = np.nanmin(np.maximum(t0, t1), axis=1)
        hit = (tmax >= np.maximum(tmin, 0.0)) & (tmin > 0)
        t = np.where(hit & (tmin < t), tmin, t)
    ok = np.isfinite(t)
    dr = np.repeat(d[ok], returns, axis=0)
    tr = np.repeat(t[ok], returns) + rng.normal(0.0, jitter, size=dr.shape[0])
    return dr * tr[:, None]


def voxelize(points, voxel=0.1, lo=(-72.0, -72.0, -2.0), hi=(72.0, 72.0, 2.0), shift=(0.0, 0.0, 0.0)):
    """Signed voxel coordinates floor((p + shift) / voxel) of the points whose
    shifted position lies inside [lo, hi) (lo, hi multiples of ``voxel``)."""
    lo = np.asarray(lo)
    hi = np.asarray(hi)
    points = points + np.asarray(shift, dtype=np.float64)
    inside = np.all((points >= lo) & (points < hi), axis=1)
    ijk = np.floor(points[inside] / voxel).astype(np.int64)
    lo_i = np.round(lo / voxel).astype(np.int64)
    hi_i = np.round(hi / voxel).astype(np.int64)
    ok = np.all((ijk >= lo_i) & (ijk < hi_i), axis=1)
    return ijk[ok].astype(np.int32)


# ---------------------------------------------------------------------------
# features / weights
# ---------------------------------------------------------------------------


def features(seed, n, c, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return rng.uniform(-1.0, 1.0, size=(n, c)).astype(np.float32)
    return rng.standard_normal(size=(n, c)).astype(np.float32)


def weights(seed, cin, cout):
    """W ~ N(0, 1/(27*cin)), layout [27, cin, cout]."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=(27, cin, cout)) * math.sqrt(1.0 / (27.0 * cin))).astype(np.float32)


# ---------------------------------------------------------------------------
# the five workloads (``scale`` < 1 gives a smaller case of the same kind)
# ---------------------------------------------------------------------------


def tiny_shell(seed=0):
    """Spherical shell, radius 24, |r - 24| <= 2, in a 64^3 box (~29k voxels).
    fp32 features U[-1,1], 16 -> 16 submanifold."""
    rng = np.random.default_rng(seed)
    out = _finish([shell_voxels()], rng)
    out.update(name="tiny_shell_64", dtype="f32", convs=[dict(cin=16, cout=16, stride=1)], feat_kind="uniform",
               seed=seed)
    return out


def leaf_dense(seed=2, scale=1.0):
    """Union of 40 solid ellipsoids (radii 8-40) in a 256^3 box; bf16 8 -> 16."""
    rng = np.random.default_rng(seed)
    box = max(16, int(round(256 * scale)))
    n = max(2, int(round(40 * scale))) if scale < 1 else 40
    v = ellipsoid_voxels(rng, box=box, n=n, rmin=8.0 * min(1.0, scale * 2), rmax=40.0 * scale)
    out = _finish([v], rng)
    out.update(name=f"leaf_dense_{box}", dtype="bf16", convs=[dict(cin=8, cout=16, stride=1)], feat_kind="normal",
               seed=seed)
    return out


def narrow_band(seed=3, scale=1.0, min_voxels=8_000_000):
    """3-voxel-wide band around a union of spheres (radii 20-150) in a 2048^3
    box; spheres are added until >= ``min_voxels``; bf16 64 -> 64."""
    rng = np.random.default_rng(seed)
    box = int(round(2048 * scale)) if scale < 1 else 2048
    rmax = 150.0 * min(1.0, scale * 4)
    rmin = min(20.0, rmax / 2)
    v = narrow_band_voxels(rng, box=box, rmin=rmin, rmax=rmax, band=1.5,
                           min_voxels=int(min_voxels * (scale ** 2 if scale < 1 else 1)))
    out = _finish([v], rng)
    out.update(name=f"narrow_band_{box}", dtype="bf16", convs=[dict(cin=64, cout=64, stride=1)],
               feat_kind="normal", seed=seed)
    return out


def lidar(seed=4, scale=1.0):
    """64 beams x 2048 azimuths, ground + 60 boxes, 5 returns per hit with
    N(0, 0.02 m) range noise, 0.1 m voxels over a 1440 x 1440 x 40 grid
    (signed coords, duplicates kept); bf16 128 -> 128 submanifold, then
    128 -> 256 stride 2.

    The grid's vertical placement is not given: its 40 voxel layers span
    [-1.85, 2.15) m around the sensor, so the ground plane (1.8 m below it)
    runs through the middle of a layer instead of along a layer boundary,
    where the noise would split every ground voxel into two layers."""
    rng = np.random.default_rng(seed)
    az = max(64, int(round(2048 * scale)))
    p = lidar_points(rng, azimuths=az)
    c = voxelize(p, shift=(0.0, 0.0, 0.05))
    out = _finish([c], rng)
    out["n_unique"] = None  # rows carry duplicates; the unique count is the build's job
    out.update(name=f"lidar_{az}az", dtype="bf16",
               convs=[dict(cin=128, cout=128, stride=1), dict(cin=128, cout=256, stride=2)],
               feat_kind="normal", seed=seed)
    return out


def batched_narrow_band(seed=5, B=8, scale=1.0, min_voxels_per_grid=1_250_000, dup_frac=0.3):
    """Batch of ``B`` narrow-band grids in 1024^3 boxes (seeds 100*seed + b),
    30% duplicate rows, rows shuffled within each batch; bf16 32 -> 64."""
    rng = np.random.default_rng(seed)
    box = int(round(1024 * scale)) if scale < 1 else 1024
    rmax = 150.0 * min(1.0, scale * 4)
    rmin = min(20.0, rmax / 2)
    per = []
    for b in range(B):
        rb = np.random.default_rng(100 * seed + b)
        per.append(narrow_band_voxels(rb, box=box, rmin=rmin, rmax=rmax, band=1.5,
                                      min_voxels=int(min_voxels_per_grid * (scale ** 2 if scale < 1 else 1))))
    out = _finish(per, rng, dup_frac=dup_frac)
    out.update(name=f"batched_narrow_band_{B}x{box}", dtype="bf16", convs=[dict(cin=32, cout=64, stride=1)],
               feat_kind="normal", seed=seed)
    return out


def ray_scene(box=1024, seed=7):
    """Narrow band (3 voxels wide) around a union of 6 spheres with centres in
    the middle of a ``box``^3 grid and radii 0.15-0.3 * box: a closed surface
    filling most of a camera's view, as the pages' 3-voxel narrow band of a
    scanned model (not available here) does."""
    rng = np.random.default_rng(seed)
    v = narrow_band_voxels(rng, box=box, rmin=0.15 * box, rmax=0.3 * box, band=1.5, n_spheres=6,
                           centre_lo=0.3, centre_hi=0.7)
    out = _finish([v], rng)
    out.update(name=f"ray_scene_{box}", seed=seed)
    return out


def camera_rays(box, n_side, seed=11, distance=1.5, half_width=0.5):
    """A pinhole camera outside a ``box``^3 grid looking at its centre:
    ``n_side``^2 rays (index space, float32) from a random direction at
    ``distance`` * box from the centre; the view spans +-half_width * box at
    the centre."""
    rng = np.random.default_rng(seed)
    c = np.full(3, box / 2.0)
    v = rng.normal(size=3)
    v /= np.linalg.norm(v)
    eye = c + v * distance * box
    fwd = -v
    up = np.array([0.0, 0.0, 1.0]) if abs(fwd[2]) < 0.9 else np.array([1.0, 0.0, 0.0])
    right = np.cross(fwd, up)
    right /= np.linalg.norm(right)
    up = np.cross(right, fwd)
    half = np.arctan(half_width / distance)  # half field of view
    u = np.tan(half) * ((np.arange(n_side) + 0.5) / n_side * 2.0 - 1.0)
    U, V = np.meshgrid(u, u, indexing="ij")
    d = fwd[None, :] + U.reshape(-1, 1) * right[None, :] + V.reshape(-1, 1) * up[None, :]
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    o = np.repeat(eye[None, :], d.shape[0], axis=0)
    return np.ascontiguousarray(o, np.float32), np.ascontiguousarray(d, np.float32)


WORKLOADS = {
    "tiny_shell": tiny_shell,
    "leaf_dense": leaf_dense,
    "narrow_band": narrow_band,
    "lidar": lidar,
    "batched_narrow_band": batched_narrow_band,
}
