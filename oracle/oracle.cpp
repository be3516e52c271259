// Plain, slow CPU oracle for the sparse-voxel hot path: IndexGrid build,
// coordinate lookup, stride-2 coarsening, 3x3x3 kernel map and sparse conv.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, imports or
// calls this file.  Only the tests, the smoke check and the benchmark's CPU
// baseline leg use it.  It shares no code, header, table or helper with the
// CUDA path; the two agree only through the written conventions below.
//
// Sources (page title + section):
//   [fVDB-notes]  "fVDB: A Deep-Learning Framework for Sparse, Large Scale, and
//                 High Performance Spatial Intelligence" (reading notes).
//                 Sections: Core method; IndexGrid; GPU-accelerated IndexGrid
//                 build; Sparse-convolution operators.
//   [DriveRT]     "DriveRT" project page, sections "Shared neighbour maps" and
//                 "Kernels selected per GPU".
//   [fVDB-ONNX]   "Proposal: ONNX Runtime support for fVDB operations",
//                 §1.1 Tensor Representations (CSR batch offsets).
//
// Conventions (the pages leave them open; these are the plainest readings):
//   * Tree: root hash -> upper node (32^3 children, covers 4096^3) -> lower
//     node (16^3 children, 128^3) -> leaf (8^3 voxels)   [fVDB-notes, Core method]
//   * Canonical voxel order: lexicographic over
//       (batch, tile_i, tile_j, tile_k, upper child (i,j,k), lower child (i,j,k),
//        voxel-in-leaf (i,j,k))
//     with tile = floor(c / 4096), upper child = (c mod 4096) div 128,
//     lower child = (c mod 128) div 8, voxel = c mod 8.  This is the depth-first
//     traversal order of the tree when root tiles are visited in signed order
//     and children in x-major bit order.
//   * Active index = 0-based rank in the canonical order; absent -> -1.
//   * Child bit n inside a node = (x * F + y) * F + z for a fanout-F node
//     (x-major); mask word = n / 64, bit = n mod 64.
//   * Leaf record = 80 bytes: 8 mask words, the index of its first active
//     voxel, and the popcounts of words 0..w-1 for w = 1..7 packed in 9-bit
//     fields (field w-1 at bit 9*(w-1)).   [fVDB-notes, IndexGrid: 80 bytes/leaf]
//   * Lower/upper nodes: child mask + per-word exclusive popcount prefix
//     (uint32) + index of the first child in the next level.
//   * Kernel offset slot s = (di+1)*9 + (dj+1)*3 + (dk+1), d in {-1,0,1}^3;
//     input coordinate of output q at slot s = stride * ijk_out(q) + d;
//     cross-correlation, no kernel flip.
//   * Conv: y[q,co] = sum_s sum_{(p,q) in list s} sum_ci x[p,ci] * W[s,ci,co],
//     accumulated in double.  A[q,co] = same sum of |x * w| (tolerance scale).
//   * Voxels along rays [fVDB-notes, HDDA]: see the definition above
//     oracle_voxels_along_rays (fp32 plane-crossing times, positive-length
//     visits of active cells, in order).
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <set>
#include <vector>
#include <algorithm>
#include <array>
#include <cmath>
#include <limits>

namespace {

// floor(a / b) for b > 0, written without relying on signed shifts.
int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b) != 0 && (a < 0)) q -= 1;
  return q;
}
// a mod b in [0, b) for b > 0.
int64_t floor_mod(int64_t a, int64_t b) { return a - b * floor_div(a, b); }

struct Voxel {
  int32_t b, i, j, k;
};

// The 13-field canonical tuple of a voxel.
std::array<int64_t, 13> canonical_tuple(const Voxel& v) {
  const int64_t c[3] = {v.i, v.j, v.k};
  std::array<int64_t, 13> t{};
  t[0] = v.b;
  for (int a = 0; a < 3; ++a) {
    int64_t tile = floor_div(c[a], 4096);
    int64_t o = floor_mod(c[a], 4096);  // offset inside the 4096^3 upper node
    t[1 + a] = tile;
    t[4 + a] = o / 128;                 // upper-node child coordinate, 0..31
    t[7 + a] = (o % 128) / 8;           // lower-node child coordinate, 0..15
    t[10 + a] = o % 8;                  // voxel inside the leaf, 0..7
  }
  return t;
}

struct CanonicalLess {
  bool operator()(const Voxel& a, const Voxel& b) const {
    return canonical_tuple(a) < canonical_tuple(b);
  }
};

// Node key: batch + node origin (coordinates rounded down to the node size).
struct NodeKey {
  int32_t b, i, j, k;
  bool operator==(const NodeKey& o) const { return b == o.b && i == o.i && j == o.j && k == o.k; }
};

NodeKey node_of(const Voxel& v, int64_t size) {
  return NodeKey{v.b, (int32_t)(v.i - floor_mod(v.i, size)), (int32_t)(v.j - floor_mod(v.j, size)),
                 (int32_t)(v.k - floor_mod(v.k, size))};
}

int popcount64(uint64_t x) {
  int c = 0;
  while (x) { x &= x - 1; ++c; }
  return c;
}

struct LeafRecord {  // 80 bytes  [fVDB-notes, IndexGrid]
  uint64_t mask[8];
  uint64_t first;
  uint64_t prefix9;
};
static_assert(sizeof(LeafRecord) == 80, "leaf record must be 80 bytes");

}  // namespace

struct oracle_grid {
  int32_t B = 0;
  int64_t n_rows = 0;
  std::map<Voxel, int64_t, CanonicalLess> index;  // coordinate -> active index
  std::vector<Voxel> voxels;                      // index -> coordinate
  std::vector<int32_t> row_to_index;              // input row -> index
  std::vector<int64_t> voxel_batch_offsets;       // CSR [B+1]
  // leaves
  std::vector<NodeKey> leaf_key;
  std::vector<LeafRecord> leaf;
  // lower nodes
  std::vector<NodeKey> lower_key;
  std::vector<uint64_t> lower_mask;    // [n_lower][64]
  std::vector<uint32_t> lower_prefix;  // [n_lower][64]
  std::vector<uint32_t> lower_first;   // first child leaf index
  // upper nodes
  std::vector<NodeKey> upper_key;
  std::vector<uint64_t> upper_mask;    // [n_upper][512]
  std::vector<uint32_t> upper_prefix;  // [n_upper][512]
  std::vector<uint32_t> upper_first;   // first child lower-node index
};

struct oracle_rays {
  std::vector<int64_t> offsets;  // [n_rays + 1]
  std::vector<int32_t> voxel;    // active index of each hit
  std::vector<float> t;          // [hits][2]: t_enter, t_exit
};

struct oracle_kmap {
  int32_t stride = 1;
  int64_t n_out = 0;
  std::vector<int64_t> offsets;  // [28]
  std::vector<int32_t> in_idx, out_idx;
  std::vector<uint32_t> out_mask;
};

namespace {

void derive_nodes(oracle_grid* g) {
  // Group active voxels (already in canonical order) into leaves, lower and
  // upper nodes.  Because the canonical order sorts by the node prefix first,
  // every node's voxels are contiguous and nodes appear in canonical order.
  const int64_t U = (int64_t)g->voxels.size();
  for (int64_t t = 0; t < U; ++t) {
    const Voxel& v = g->voxels[t];
    NodeKey lk = node_of(v, 8), wk = node_of(v, 128), uk = node_of(v, 4096);
    if (g->upper_key.empty() || !(g->upper_key.back() == uk)) {
      g->upper_key.push_back(uk);
      g->upper_mask.resize(g->upper_key.size() * 512, 0);
      g->upper_first.push_back((uint32_t)g->lower_key.size());
    }
    if (g->lower_key.empty() || !(g->lower_key.back() == wk)) {
      g->lower_key.push_back(wk);
      g->lower_mask.resize(g->lower_key.size() * 64, 0);
      g->lower_first.push_back((uint32_t)g->leaf_key.size());
      // register the new lower node in its upper node
      int64_t n = ((floor_mod(v.i, 4096) / 128) * 32 + floor_mod(v.j, 4096) / 128) * 32 + floor_mod(v.k, 4096) / 128;
      g->upper_mask[(g->upper_key.size() - 1) * 512 + n / 64] |= (uint64_t)1 << (n % 64);
    }
    if (g->leaf_key.empty() || !(g->leaf_key.back() == lk)) {
      g->leaf_key.push_back(lk);
      LeafRecord r{};
      r.first = (uint64_t)t;
      g->leaf.push_back(r);
      int64_t n = (((floor_mod(v.i, 128) / 8) * 16 + floor_mod(v.j, 128) / 8) * 16) + floor_mod(v.k, 128) / 8;
      g->lower_mask[(g->lower_key.size() - 1) * 64 + n / 64] |= (uint64_t)1 << (n % 64);
    }
    int64_t n = (floor_mod(v.i, 8) * 8 + floor_mod(v.j, 8)) * 8 + floor_mod(v.k, 8);
    g->leaf.back().mask[n / 64] |= (uint64_t)1 << (n % 64);
  }
  // prefix popcounts
  for (auto& r : g->leaf) {
    uint64_t acc = 0, packed = 0;
    for (int w = 1; w < 8; ++w) {
      acc += (uint64_t)popcount64(r.mask[w - 1]);
      packed |= acc << (9 * (w - 1));
    }
    r.prefix9 = packed;
  }
  g->lower_prefix.assign(g->lower_key.size() * 64, 0);
  for (size_t a = 0; a < g->lower_key.size(); ++a) {
    uint32_t acc = 0;
    for (int w = 0; w < 64; ++w) {
      g->lower_prefix[a * 64 + w] = acc;
      acc += (uint32_t)popcount64(g->lower_mask[a * 64 + w]);
    }
  }
  g->upper_prefix.assign(g->upper_key.size() * 512, 0);
  for (size_t a = 0; a < g->upper_key.size(); ++a) {
    uint32_t acc = 0;
    for (int w = 0; w < 512; ++w) {
      g->upper_prefix[a * 512 + w] = acc;
      acc += (uint32_t)popcount64(g->upper_mask[a * 512 + w]);
    }
  }
}

oracle_grid* build_from_voxel_rows(const std::vector<Voxel>& rows, int32_t B) {
  oracle_grid* g = new oracle_grid();
  g->B = B;
  g->n_rows = (int64_t)rows.size();
  // 1. unique coordinates in canonical order (std::map does both).
  for (const Voxel& v : rows) g->index.emplace(v, 0);
  // 2. index = rank in canonical order.
  int64_t t = 0;
  g->voxels.reserve(g->index.size());
  for (auto& kv : g->index) {
    kv.second = t++;
    g->voxels.push_back(kv.first);
  }
  // 3. every input row (duplicates included) maps to the index of its voxel.
  g->row_to_index.resize(rows.size());
  for (size_t r = 0; r < rows.size(); ++r) g->row_to_index[r] = (int32_t)g->index.at(rows[r]);
  // 4. per-batch voxel ranges: batch is the most significant order field.
  g->voxel_batch_offsets.assign((size_t)B + 1, 0);
  for (const Voxel& v : g->voxels) g->voxel_batch_offsets[(size_t)v.b + 1] += 1;
  for (int32_t b = 0; b < B; ++b) g->voxel_batch_offsets[b + 1] += g->voxel_batch_offsets[b];
  derive_nodes(g);
  return g;
}

}  // namespace

extern "C" {

int32_t oracle_leaf_record_bytes(void) { return (int32_t)sizeof(LeafRecord); }

// Build from int32 coords [n_rows,3] and CSR row offsets [B+1].
// [fVDB-notes, GPU-accelerated IndexGrid build] computes the same set of
// active voxels and the same tree; here by std::map, in canonical order.
// Returns nullptr on malformed offsets.
oracle_grid* oracle_build(const int32_t* coords, int64_t n_rows, const int64_t* batch_offsets, int32_t B) {
  if (B < 1 || n_rows < 0 || batch_offsets[0] != 0 || batch_offsets[B] != n_rows) return nullptr;
  std::vector<Voxel> rows((size_t)n_rows);
  for (int32_t b = 0; b < B; ++b) {
    if (batch_offsets[b + 1] < batch_offsets[b]) return nullptr;
    for (int64_t r = batch_offsets[b]; r < batch_offsets[b + 1]; ++r)
      rows[(size_t)r] = Voxel{b, coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]};
  }
  return build_from_voxel_rows(rows, B);
}

void oracle_grid_free(oracle_grid* g) { delete g; }

// counts[0..3] = n_upper, n_lower, n_leaf, n_active
void oracle_grid_counts(const oracle_grid* g, int64_t* counts) {
  counts[0] = (int64_t)g->upper_key.size();
  counts[1] = (int64_t)g->lower_key.size();
  counts[2] = (int64_t)g->leaf_key.size();
  counts[3] = (int64_t)g->voxels.size();
}

int64_t oracle_grid_rows(const oracle_grid* g) { return g->n_rows; }

// ijk [U,3], batch [U], row_to_index [n_rows], voxel_batch_offsets [B+1]
void oracle_grid_voxels(const oracle_grid* g, int32_t* ijk, int32_t* batch, int32_t* row_to_index,
                        int64_t* voxel_batch_offsets) {
  for (size_t t = 0; t < g->voxels.size(); ++t) {
    ijk[3 * t] = g->voxels[t].i;
    ijk[3 * t + 1] = g->voxels[t].j;
    ijk[3 * t + 2] = g->voxels[t].k;
    batch[t] = g->voxels[t].b;
  }
  std::memcpy(row_to_index, g->row_to_index.data(), g->row_to_index.size() * sizeof(int32_t));
  std::memcpy(voxel_batch_offsets, g->voxel_batch_offsets.data(), g->voxel_batch_offsets.size() * sizeof(int64_t));
}

// origin [L,3], batch [L], records [L] as 10 uint64 each (mask[8], first, prefix9)
void oracle_grid_leaves(const oracle_grid* g, int32_t* origin, int32_t* batch, uint64_t* records) {
  for (size_t a = 0; a < g->leaf_key.size(); ++a) {
    origin[3 * a] = g->leaf_key[a].i;
    origin[3 * a + 1] = g->leaf_key[a].j;
    origin[3 * a + 2] = g->leaf_key[a].k;
    batch[a] = g->leaf_key[a].b;
    std::memcpy(records + 10 * a, &g->leaf[a], sizeof(LeafRecord));
  }
}

// origin [n,3], batch [n], mask [n,64], prefix [n,64], first_leaf [n]
void oracle_grid_lower(const oracle_grid* g, int32_t* origin, int32_t* batch, uint64_t* mask, uint32_t* prefix,
                       uint32_t* first_leaf) {
  for (size_t a = 0; a < g->lower_key.size(); ++a) {
    origin[3 * a] = g->lower_key[a].i;
    origin[3 * a + 1] = g->lower_key[a].j;
    origin[3 * a + 2] = g->lower_key[a].k;
    batch[a] = g->lower_key[a].b;
  }
  std::memcpy(mask, g->lower_mask.data(), g->lower_mask.size() * 8);
  std::memcpy(prefix, g->lower_prefix.data(), g->lower_prefix.size() * 4);
  std::memcpy(first_leaf, g->lower_first.data(), g->lower_first.size() * 4);
}

// origin [n,3], batch [n], mask [n,512], prefix [n,512], first_lower [n]
void oracle_grid_upper(const oracle_grid* g, int32_t* origin, int32_t* batch, uint64_t* mask, uint32_t* prefix,
                       uint32_t* first_lower) {
  for (size_t a = 0; a < g->upper_key.size(); ++a) {
    origin[3 * a] = g->upper_key[a].i;
    origin[3 * a + 1] = g->upper_key[a].j;
    origin[3 * a + 2] = g->upper_key[a].k;
    batch[a] = g->upper_key[a].b;
  }
  std::memcpy(mask, g->upper_mask.data(), g->upper_mask.size() * 8);
  std::memcpy(prefix, g->upper_prefix.data(), g->upper_prefix.size() * 4);
  std::memcpy(first_lower, g->upper_first.data(), g->upper_first.size() * 4);
}

// Coordinate -> active index or -1 (map lookup).  [fVDB-ONNX §1.2: IJKToIndex]
void oracle_lookup(const oracle_grid* g, const int32_t* coords, const int32_t* batch, int64_t n, int32_t* out) {
  for (int64_t r = 0; r < n; ++r) {
    Voxel v{batch[r], coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]};
    auto it = g->index.find(v);
    out[r] = (it == g->index.end()) ? -1 : (int32_t)it->second;
  }
}

// Output grid of a stride-s conv: unique floor(ijk / s) of the active voxels,
// per batch.  [fVDB-ONNX §1.2: CoarsenedGrid / ConvGrid]
oracle_grid* oracle_coarsen(const oracle_grid* g, int32_t stride) {
  if (stride < 1) return nullptr;
  std::vector<Voxel> rows;
  rows.reserve(g->voxels.size());
  for (const Voxel& v : g->voxels)
    rows.push_back(Voxel{v.b, (int32_t)floor_div(v.i, stride), (int32_t)floor_div(v.j, stride),
                         (int32_t)floor_div(v.k, stride)});
  return build_from_voxel_rows(rows, g->B);
}

// Refined grid: every voxel's factor^3 children, factor * ijk + (0..factor-1)^3,
// per batch.  [fVDB-ONNX, §1.2 Grid-to-Grid ops: RefinedGrid]
oracle_grid* oracle_refine(const oracle_grid* g, int32_t factor) {
  if (factor < 1) return nullptr;
  std::vector<Voxel> rows;
  rows.reserve(g->voxels.size() * (size_t)factor * factor * factor);
  for (const Voxel& v : g->voxels)
    for (int a = 0; a < factor; ++a)
      for (int b = 0; b < factor; ++b)
        for (int c = 0; c < factor; ++c)
          rows.push_back(Voxel{v.b, (int32_t)((int64_t)factor * v.i + a), (int32_t)((int64_t)factor * v.j + b),
                               (int32_t)((int64_t)factor * v.k + c)});
  return build_from_voxel_rows(rows, g->B);
}

// A coordinate a grid can hold.  Neighbour positions are computed exactly in
// 64 bits; one outside int32 is no voxel of any grid (no wrap-around).
static bool in_int32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

// 3x3x3 kernel map: for every output voxel q (ascending) and offset slot s,
// look up the input voxel at stride*ijk_out(q) + d_s in the same batch.
// [DriveRT, Shared neighbour maps]; mask bit s set when the pair exists
// [DriveRT, Kernels selected per GPU].
oracle_kmap* oracle_kernel_map(const oracle_grid* gin, const oracle_grid* gout, int32_t stride) {
  if (stride != 1 && stride != 2) return nullptr;
  oracle_kmap* m = new oracle_kmap();
  m->stride = stride;
  m->n_out = (int64_t)gout->voxels.size();
  m->out_mask.assign((size_t)m->n_out, 0);
  std::vector<std::vector<int32_t>> lin(27), lout(27);
  for (int64_t q = 0; q < m->n_out; ++q) {
    const Voxel& o = gout->voxels[q];
    for (int di = -1; di <= 1; ++di)
      for (int dj = -1; dj <= 1; ++dj)
        for (int dk = -1; dk <= 1; ++dk) {
          int s = (di + 1) * 9 + (dj + 1) * 3 + (dk + 1);
          const int64_t ci = (int64_t)stride * o.i + di, cj = (int64_t)stride * o.j + dj,
                        ck = (int64_t)stride * o.k + dk;
          if (!in_int32(ci) || !in_int32(cj) || !in_int32(ck)) continue;  // no such voxel: no pair
          Voxel c{o.b, (int32_t)ci, (int32_t)cj, (int32_t)ck};
          auto it = gin->index.find(c);
          if (it != gin->index.end()) {
            lin[s].push_back((int32_t)it->second);
            lout[s].push_back((int32_t)q);
            m->out_mask[q] |= 1u << s;
          }
        }
  }
  m->offsets.assign(28, 0);
  for (int s = 0; s < 27; ++s) m->offsets[s + 1] = m->offsets[s] + (int64_t)lin[s].size();
  for (int s = 0; s < 27; ++s) {
    m->in_idx.insert(m->in_idx.end(), lin[s].begin(), lin[s].end());
    m->out_idx.insert(m->out_idx.end(), lout[s].begin(), lout[s].end());
  }
  return m;
}

void oracle_kmap_free(oracle_kmap* m) { delete m; }
int64_t oracle_kmap_pairs(const oracle_kmap* m) { return m->offsets[27]; }

void oracle_kmap_export(const oracle_kmap* m, int64_t* offsets, int32_t* in_idx, int32_t* out_idx, uint32_t* mask) {
  std::memcpy(offsets, m->offsets.data(), 28 * sizeof(int64_t));
  std::memcpy(in_idx, m->in_idx.data(), m->in_idx.size() * 4);
  std::memcpy(out_idx, m->out_idx.data(), m->out_idx.size() * 4);
  std::memcpy(mask, m->out_mask.data(), m->out_mask.size() * 4);
}

// Sparse conv over the kernel map, in double:
//   y[q,co] = sum_s sum_{(p,q) in list s} sum_ci x[p,ci] * W[s,ci,co]
//   a[q,co] = the same sum of |x[p,ci] * W[s,ci,co]|
// x: [n_in, cin], W: [27, cin, cout], y/a: [n_out, cout], row-major doubles.
// [fVDB-notes, Sparse-convolution operators: gather-GEMM-scatter]
// Kernel map of the transposed convolution: for every output voxel p of gout
// (ascending) and slot s, the input voxel q of gin with stride * ijk(q) + d_s =
// ijk(p) in the same batch, i.e. q = (ijk(p) - d_s) / stride when that division
// is exact.  [fVDB-ONNX, §1.2 Grid-to-Grid ops: ConvTransposeGrid]  Its pairs are
// those of oracle_kernel_map(gout, gin, stride) with input and output swapped.
oracle_kmap* oracle_kernel_map_transposed(const oracle_grid* gin, const oracle_grid* gout, int32_t stride) {
  if (stride != 1 && stride != 2) return nullptr;
  oracle_kmap* m = new oracle_kmap();
  m->stride = stride;
  m->n_out = (int64_t)gout->voxels.size();
  m->out_mask.assign((size_t)m->n_out, 0);
  std::vector<std::vector<int32_t>> lin(27), lout(27);
  for (int64_t p = 0; p < m->n_out; ++p) {
    const Voxel& o = gout->voxels[p];
    for (int di = -1; di <= 1; ++di)
      for (int dj = -1; dj <= 1; ++dj)
        for (int dk = -1; dk <= 1; ++dk) {
          const int s = (di + 1) * 9 + (dj + 1) * 3 + (dk + 1);
          const int64_t ci = (int64_t)o.i - di, cj = (int64_t)o.j - dj, ck = (int64_t)o.k - dk;
          if (ci % stride != 0 || cj % stride != 0 || ck % stride != 0) continue;
          if (!in_int32(ci / stride) || !in_int32(cj / stride) || !in_int32(ck / stride)) continue;
          Voxel c{o.b, (int32_t)(ci / stride), (int32_t)(cj / stride), (int32_t)(ck / stride)};
          auto it = gin->index.find(c);
          if (it != gin->index.end()) {
            lin[s].push_back((int32_t)it->second);
            lout[s].push_back((int32_t)p);
            m->out_mask[p] |= 1u << s;
          }
        }
  }
  m->offsets.assign(28, 0);
  for (int s = 0; s < 27; ++s) m->offsets[s + 1] = m->offsets[s] + (int64_t)lin[s].size();
  for (int s = 0; s < 27; ++s) {
    m->in_idx.insert(m->in_idx.end(), lin[s].begin(), lin[s].end());
    m->out_idx.insert(m->out_idx.end(), lout[s].begin(), lout[s].end());
  }
  return m;
}

// Weight gradient: dW[s][ci][co] = sum over the pairs (p, q) of list s of
// x[p][ci] * dy[q][co], in double.  [fVDB-notes, Sparse-convolution operators:
// training computes gradients through the general (pair-list) backend]
void oracle_conv_wgrad(const oracle_kmap* m, const double* x, int64_t cin, const double* dy, int64_t cout,
                       double* dW) {
  std::memset(dW, 0, sizeof(double) * (size_t)(27 * cin * cout));
  for (int s = 0; s < 27; ++s) {
    double* Ws = dW + (size_t)s * cin * cout;
    for (int64_t e = m->offsets[s]; e < m->offsets[s + 1]; ++e) {
      const double* xp = x + (size_t)m->in_idx[e] * cin;
      const double* gq = dy + (size_t)m->out_idx[e] * cout;
      for (int64_t ci = 0; ci < cin; ++ci)
        for (int64_t co = 0; co < cout; ++co) Ws[ci * cout + co] += xp[ci] * gq[co];
    }
  }
}

void oracle_conv(const oracle_kmap* m, const double* x, int64_t cin, const double* W, int64_t cout, double* y,
                 double* a) {
  std::memset(y, 0, sizeof(double) * (size_t)(m->n_out * cout));
  std::memset(a, 0, sizeof(double) * (size_t)(m->n_out * cout));
  for (int s = 0; s < 27; ++s) {
    const double* Ws = W + (size_t)s * cin * cout;
    for (int64_t e = m->offsets[s]; e < m->offsets[s + 1]; ++e) {
      const double* xp = x + (size_t)m->in_idx[e] * cin;
      double* yq = y + (size_t)m->out_idx[e] * cout;
      double* aq = a + (size_t)m->out_idx[e] * cout;
      for (int64_t ci = 0; ci < cin; ++ci)
        for (int64_t co = 0; co < cout; ++co) {
          double t = xp[ci] * Ws[ci * cout + co];
          yq[co] += t;
          aq[co] += (t < 0 ? -t : t);
        }
    }
  }
}

// The same sum for a chosen set of output rows only (sampled checks at sizes
// where the full conv is too slow).  Uses the map lookups directly, so it needs
// no kernel map: rows[r] is an output index of gout.
void oracle_conv_rows(const oracle_grid* gin, const oracle_grid* gout, int32_t stride, const int64_t* rows,
                      int64_t n_rows, const double* x, int64_t cin, const double* W, int64_t cout, double* y,
                      double* a) {
  std::memset(y, 0, sizeof(double) * (size_t)(n_rows * cout));
  std::memset(a, 0, sizeof(double) * (size_t)(n_rows * cout));
  for (int64_t r = 0; r < n_rows; ++r) {
    const Voxel& o = gout->voxels[(size_t)rows[r]];
    for (int di = -1; di <= 1; ++di)
      for (int dj = -1; dj <= 1; ++dj)
        for (int dk = -1; dk <= 1; ++dk) {
          int s = (di + 1) * 9 + (dj + 1) * 3 + (dk + 1);
          const int64_t pi = (int64_t)stride * o.i + di, pj = (int64_t)stride * o.j + dj,
                        pk = (int64_t)stride * o.k + dk;
          if (!in_int32(pi) || !in_int32(pj) || !in_int32(pk)) continue;  // no such voxel: no pair
          Voxel c{o.b, (int32_t)pi, (int32_t)pj, (int32_t)pk};
          auto it = gin->index.find(c);
          if (it == gin->index.end()) continue;
          const double* xp = x + (size_t)it->second * cin;
          const double* Ws = W + (size_t)s * cin * cout;
          for (int64_t ci = 0; ci < cin; ++ci)
            for (int64_t co = 0; co < cout; ++co) {
              double t = xp[ci] * Ws[ci * cout + co];
              y[r * cout + co] += t;
              a[r * cout + co] += (t < 0 ? -t : t);
            }
        }
  }
}

}  // extern "C"

// ---------------------------------------------------------------- voxels along rays
// [fVDB-notes, HDDA] marches rays through the grid with one DDA per tree level
// so that empty nodes are crossed in one step; what it yields is the voxels
// each ray passes through.  This oracle gets the same voxels the slow way: one
// per-voxel DDA that steps through every cell and asks the map whether the
// cell is active.
//
// Definition (written out here and in the CUDA source; the two share no code):
//   * voxel (i,j,k) is the cell [i,i+1) x [j,j+1) x [k,k+1) in index space;
//     the ray is o + t d with fp32 o, d; inv_a = 1 / d_a (fp32, rounded once).
//   * The ray crosses the plane x_a = n at T_a(n) = ((float)n - o_a) * inv_a,
//     two fp32 operations each rounded to nearest (no fused multiply-add).
//   * [tmin, tmax] is clipped to the bounding box [lo, hi + 1) of the batch
//     element's active voxels by the same plane times (slab method); a
//     direction component of 0 keeps the ray only if lo_a <= o_a < hi_a + 1;
//     d = 0 or an empty clip gives no hits.
//   * At time t the ray is in cell c_a = max{n : T_a(n) <= t} (d_a > 0),
//     min{n : T_a(n) <= t} - 1 (d_a < 0), floor(o_a) (d_a = 0).
//   * A hit is an active cell the ray occupies for a time interval of
//     positive length inside the clipped segment [t0, t1): its index and
//     [t_enter, t_exit) = the times of the crossings that enter and leave it,
//     clipped to [t0, t1).  Hits come in order of t_enter.
// Any box holding all active voxels gives the same hits (cells outside hold
// none, and a hit's entry crossing is never before the box's), so the CUDA
// path may clip to a larger box.
namespace {

float plane_time(int64_t n, float o, float inv) {
  const float diff = (float)n - o;
  return diff * inv;
}

// Cell coordinate along one axis at time t (definition above).
int64_t cell_at(float o, float d, float inv, float t) {
  if (d > 0.0f) {
    int64_t n = (int64_t)std::floor((double)o + (double)t * (double)d);
    while (plane_time(n + 1, o, inv) <= t) ++n;
    while (plane_time(n, o, inv) > t) --n;
    return n;
  }
  if (d < 0.0f) {
    int64_t m = (int64_t)std::floor((double)o + (double)t * (double)d) + 1;
    while (plane_time(m - 1, o, inv) <= t) --m;
    while (plane_time(m, o, inv) > t) ++m;
    return m - 1;
  }
  return (int64_t)std::floor((double)o);
}

void march_one(const oracle_grid* g, const int64_t* lo, const int64_t* hi, int32_t b, const float* o,
               const float* d, float tmin, float tmax, oracle_rays* out) {
  if (d[0] == 0.0f && d[1] == 0.0f && d[2] == 0.0f) return;
  float inv[3];
  float t0 = tmin, t1 = tmax;
  for (int a = 0; a < 3; ++a) {
    if (d[a] == 0.0f) {
      inv[a] = 0.0f;
      if (o[a] < (float)lo[a] || o[a] >= (float)(hi[a] + 1)) return;
      continue;
    }
    inv[a] = 1.0f / d[a];
    float ta = plane_time(lo[a], o[a], inv[a]), tb = plane_time(hi[a] + 1, o[a], inv[a]);
    if (ta > tb) std::swap(ta, tb);
    t0 = std::max(t0, ta);
    t1 = std::min(t1, tb);
  }
  if (!(t0 < t1)) return;
  int64_t c[3];
  float next[3];
  const float inf = std::numeric_limits<float>::infinity();
  for (int a = 0; a < 3; ++a) {
    c[a] = cell_at(o[a], d[a], inv[a], t0);
    next[a] = d[a] > 0.0f ? plane_time(c[a] + 1, o[a], inv[a]) : d[a] < 0.0f ? plane_time(c[a], o[a], inv[a]) : inf;
  }
  float enter = t0;
  for (;;) {
    const float T = std::min(next[0], std::min(next[1], next[2]));
    const float exit = std::min(T, t1);
    if (exit > enter) {
      auto it = g->index.find(Voxel{b, (int32_t)c[0], (int32_t)c[1], (int32_t)c[2]});
      if (it != g->index.end()) {
        out->voxel.push_back((int32_t)it->second);
        out->t.push_back(enter);
        out->t.push_back(exit);
      }
    }
    if (T >= t1) break;
    for (int a = 0; a < 3; ++a) {
      if (next[a] != T) continue;
      if (d[a] > 0.0f) {
        c[a] += 1;
        next[a] = plane_time(c[a] + 1, o[a], inv[a]);
      } else {
        c[a] -= 1;
        next[a] = plane_time(c[a], o[a], inv[a]);
      }
    }
    enter = T;
  }
}

}  // namespace

extern "C" {

// Rays [n][3] origins and directions (index space, fp32), batch element of
// each ray (NULL: all 0), one segment [tmin, tmax] for all.  Returns the hits
// in CSR form (see the definition above); nullptr for a batch out of range.
oracle_rays* oracle_voxels_along_rays(const oracle_grid* g, const float* origins, const float* dirs,
                                      const int32_t* batch, int64_t n, float tmin, float tmax) {
  std::vector<int64_t> lo((size_t)g->B * 3, 0), hi((size_t)g->B * 3, 0);
  std::vector<char> any((size_t)g->B, 0);
  for (const Voxel& v : g->voxels) {
    const int64_t c[3] = {v.i, v.j, v.k};
    for (int a = 0; a < 3; ++a) {
      int64_t& l = lo[(size_t)v.b * 3 + a];
      int64_t& h = hi[(size_t)v.b * 3 + a];
      if (!any[(size_t)v.b] || c[a] < l) l = c[a];
      if (!any[(size_t)v.b] || c[a] > h) h = c[a];
    }
    any[(size_t)v.b] = 1;
  }
  oracle_rays* r = new oracle_rays();
  r->offsets.push_back(0);
  for (int64_t q = 0; q < n; ++q) {
    const int32_t b = batch ? batch[q] : 0;
    if (b < 0 || b >= g->B) {
      delete r;
      return nullptr;
    }
    if (any[(size_t)b])
      march_one(g, &lo[(size_t)b * 3], &hi[(size_t)b * 3], b, origins + 3 * q, dirs + 3 * q, tmin, tmax, r);
    r->offsets.push_back((int64_t)r->voxel.size());
  }
  return r;
}

int64_t oracle_rays_hits(const oracle_rays* r) { return (int64_t)r->voxel.size(); }

void oracle_rays_export(const oracle_rays* r, int64_t* offsets, int32_t* voxel, float* t) {
  std::memcpy(offsets, r->offsets.data(), r->offsets.size() * 8);
  std::memcpy(voxel, r->voxel.data(), r->voxel.size() * 4);
  std::memcpy(t, r->t.data(), r->t.size() * 4);
}

void oracle_rays_free(oracle_rays* r) { delete r; }

}  // extern "C"
