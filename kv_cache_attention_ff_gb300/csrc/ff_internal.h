// Structures shared by the host side of libff (ff_bank.cpp) and its kernels.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ff {

// ------------------------------------------------------------------ G1 / G2
// One launch of the RoPE + publish kernel processes a list of frame-sized work
// items.  Every item covers one latent frame of one (K, V) pair,
// T * heads * head_dim bf16 each, split into 16-byte units; a thread handles
// the same unit offsets of whatever an item touches (one unit of G consecutive
// heads of a token, sharing their rotary angles).  An item reads a K and a V
// frame, rotates K under the published-K contract and writes both to their
// destination frames (a stage-ring slot, an anchor slot or a scratch buffer);
// with src_q set it also rotates that Q frame into dst_q.

struct G1Item {
  const void* src_k;  // K frame before rotary encoding
  const void* src_v;  // V frame
  const void* src_q;  // Q frame before rotary encoding, or null
  void* dst_k;        // rotated K frame
  void* dst_v;        // V frame (copied)
  void* dst_q;        // rotated Q frame (when src_q is set)
  int t;              // absolute latent frame (rotary time position)
};

constexpr int kMaxItems = 160;
constexpr int kFewItems = 8;  // launches with at most this many items use a small parameter block
constexpr int kBatchItems = 32;  // a batch of renderer calls: at most 4 calls x 8 frames

struct G1Header {
  const double2* rope64;  // rotary (cos, sin) in fp64: [total_frames][pt], then [frame_h][py], then [frame_w][px]
  const float2* rope32;   // the same table rounded to fp32
  int y_base, x_base;     // first row-axis and column-axis entries
  long long units_per_frame;  // T * h * d / 8
  int units_per_row;          // h * d / 8  (16-byte units per token)
  int units_per_head;         // d / 8 (a power of two)
  int frame_w;
  float inv_frame_w;          // fp32 reciprocal for the token -> (row, column) division
  int pt, py;                 // channel pairs on the time and row axes (pairs beyond pt+py: column axis)
  int px;
  int n_items;
};

template <int N>
struct G1ParamsN : G1Header {
  static constexpr int kItems = N;
  G1Item items[N];
};
using G1Params = G1ParamsN<kMaxItems>;

// ----------------------------------------------------------------- attention

// Attention work is described as query groups, each a run of query rows with
// its own list of key segments and its own output.  A segment is a row range
// of one of the K/V tensor-map pairs the launch carries.  A renderer call is
// one group whose segments are read in place: runs of adjacent anchor slots and
// runs of adjacent stage-ring slots, each with its own map whose extent ends at
// the segment (rows past it read as zeros).  A batch of independent renderer
// calls is one group per call; a planner call adds its own block from scratch;
// a packed block-causal forward has one group per chunk, all segments in one
// workspace map.
constexpr int kMaxGroups = 96;
constexpr int kMaxSegs = 4;
constexpr int kMaxMaps = 4;
constexpr int kMaxSplit = 4;  // key ranges a split unit is cut into, at most
constexpr int kMaxBatch = 4;  // renderer calls in one batched launch

struct AttnGroup {
  int q_row0;              // first query row of the group
  int nq;                  // query rows
  int qb0;                 // first linear 256-row query block of the group
  int n_seg;               // key segments (1..kMaxSegs)
  int seg_map[kMaxSegs];   // K/V map pair of each segment
  int seg_row0[kMaxSegs];  // first key row of each segment within its map
  int seg_rows[kMaxSegs];  // key rows of each segment
  int seg_tile0[kMaxSegs]; // first 128-key tile of each segment in the group's tile sequence
  int n_kv;                // tiles over all segments
  int out_row0;            // row of `out` that query row q_row0 goes to
  void* out;               // bf16 [rows, h, d] output of the group
};

// K and V tensor maps of a launch (bf16 [rows, heads * head_dim], 64 x 128 boxes).
template <int M>
struct KVMapsN {
  static constexpr int kMaps = M;
  CUtensorMap k[M];
  CUtensorMap v[M];
};
using KVMaps = KVMapsN<kMaxMaps>;
using KVMapsBatch = KVMapsN<kMaxMaps * kMaxBatch>;

struct AttnHeader {
  float* part_o;        // [split pieces][256][d] unnormalised partial outputs
  float* part_ml;       // [split pieces][256][2] running max (log2 units) and sum
  unsigned int* err;    // device error word
  int heads;
  int n_qb;             // linear 256-row query blocks over all groups
  // Work units are (head, linear query block), u = head * n_qb + block.  Units
  // 0 .. n_whole-1 are one piece each (their whole key range, output written
  // directly); the others are cut into n_split key ranges whose partials the
  // combine kernel merges.  Pieces: the whole units in order, then the split
  // pieces ordered (split, unit).
  int n_whole;
  int n_split;          // key ranges per split unit (1: every unit is whole)
  int n_pieces;         // n_whole + (heads * n_qb - n_whole) * n_split
  float scale_log2;     // log2(e) / sqrt(d)
  int n_groups;
};

// Kernel parameters with room for NG query groups; launches with one group
// (every renderer and planner call) use NG = 1, which keeps the parameter
// block small.
template <int NG>
struct AttnParamsN : AttnHeader {
  AttnGroup groups[NG];
};
using AttnParams = AttnParamsN<kMaxGroups>;

// Fill `p` with the single group [0, nq) x one key segment [0, nk) of map 0,
// output rows [0, nq) of `out`.
inline void attn_single_group(AttnParams& p, int nq, int nk, void* out) {
  p.n_groups = 1;
  AttnGroup& g = p.groups[0];
  g.q_row0 = 0;
  g.nq = nq;
  g.qb0 = 0;
  g.n_seg = 1;
  g.seg_map[0] = 0;
  g.seg_row0[0] = 0;
  g.seg_rows[0] = nk;
  g.seg_tile0[0] = 0;
  g.n_kv = (nk + 127) / 128;
  g.out = out;
  g.out_row0 = 0;
  p.n_qb = (nq + 255) / 256;
}

// Work plan of an attention call with `units` (head, query block) units of
// n_kv key tiles on `sms` persistent CTAs: the first n_whole units run as one
// piece each, the others as n_split key ranges merged by the combine kernel.
// Candidates are whole waves of whole units followed by split units (and the
// plan with no split at all, which needs no partials); each is scored by the
// round-robin makespan in tiles (+2 per piece for its prologue and epilogue)
// plus the combine's cost (about 1e-4 tile per partial row).  Split plans
// whose partials exceed max_part_rows rows are not considered.
struct SplitPlan {
  int n_whole, n_split, n_pieces;
  size_t part_rows;
};

inline SplitPlan plan_split(int units, int n_kv, int sms, size_t max_part_rows) {
  SplitPlan best{units, 1, units, 0};
  double best_cost = 1e300;
  std::vector<double> load(static_cast<size_t>(std::max(sms, 1)));
  for (int ns = 1; ns <= std::min(kMaxSplit, n_kv); ++ns) {
    for (int m = 0; m * sms <= units; ++m) {
      const int n_whole = (ns == 1) ? units : m * sms;
      const int rest = units - n_whole;
      if (ns > 1 && rest == 0) continue;
      const size_t rows = static_cast<size_t>(rest) * ns * 256;
      if (ns > 1 && rows > max_part_rows) continue;
      const int pieces = n_whole + rest * ns;
      const int grid = std::min(pieces, sms);
      std::fill(load.begin(), load.begin() + grid, 0.0);
      for (int pc = 0; pc < pieces; ++pc) {
        int tiles = n_kv;
        if (pc >= n_whole) {
          const int split = (pc - n_whole) / rest;
          tiles = static_cast<int>((static_cast<long long>(split + 1) * n_kv) / ns -
                                   (static_cast<long long>(split) * n_kv) / ns);
        }
        load[pc % grid] += tiles + 2.0;
      }
      double cost = *std::max_element(load.begin(), load.begin() + grid);
      if (ns > 1) cost += 4.0 + static_cast<double>(rows) * 1e-4;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = {n_whole, ns, pieces, ns > 1 ? rows : 0};
      }
      if (ns == 1) break;
    }
  }
  return best;
}

// Host launchers (ff_publish.cu / ff_attn.cu).
cudaError_t launch_publish(const G1Params& p, int grid, cudaStream_t s);
cudaError_t launch_attention(int head_dim, const CUtensorMap& tq, const KVMaps& kv, const AttnParams& p, int grid,
                             cudaStream_t s);
// A batch launch: at most kMaxBatch groups over up to kMaxMaps * kMaxBatch map pairs.
cudaError_t launch_attention(int head_dim, const CUtensorMap& tq, const KVMapsBatch& kv, const AttnParams& p,
                             int grid, cudaStream_t s);
cudaError_t launch_combine(int head_dim, const AttnParams& p, cudaStream_t s);
size_t attention_smem_bytes(int head_dim);
cudaError_t launch_wait_probe(unsigned int* err, unsigned long long limit_ns, cudaStream_t s);
cudaError_t attention_configure(int head_dim);


}  // namespace ff
