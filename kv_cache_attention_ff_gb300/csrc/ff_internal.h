// Structures shared by the host side of libff (ff_bank.cpp) and its kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ff {

// ------------------------------------------------------------------ G1 / G2
// One launch of the RoPE + publish + gather kernel processes a list of
// frame-sized work items.  Every item covers one latent frame of one
// tensor pair (K and V), T * heads * head_dim bf16 each, split into 16-byte
// units; a thread handles the same unit offset of whatever an item touches.

enum ItemKind : int {
  kItemCopy = 0,    // context frame <- (k, v) source frame (anchor or history slot)
  kItemOwn = 1,     // own chunk frame r: RoPE(q) -> q_rot, RoPE(k) and v -> slot frame r and context
  kItemAnchor = 2,  // anchor input frame r: RoPE(k) and v -> anchor slot
  kItemOwnCtx = 3,  // like kItemOwn but nothing is published (planner blocks, packed frames)
  kItemRotCtx = 4,  // context frame <- (RoPE(k), v) of the source frame in (k, v); no Q, nothing published
};

struct G1Item {
  const void* k;   // copy: source K frame; own/anchor: destination K frame (slot)
  const void* v;   // same for V
  int kind;
  int ctx;         // copy/own: context frame written (-1: none)
  int r;           // own/anchor: frame index in the call's inputs
  int t;           // own/anchor: absolute latent frame (rotary time position)
  int old_ctx;     // own: context frame that receives the slot's previous content
                   // before it is overwritten (-1: nothing to save)
  int pad;
};

constexpr int kMaxItems = 160;

struct G1Params {
  const void* q_in;   // own chunk inputs [F * T, h, d] (q unused for anchors)
  const void* k_in;
  const void* v_in;
  void* q_rot;        // [F * T, h, d]
  void* ctx_k;        // [key_frames * T, h, d]
  void* ctx_v;
  const double2* rope64;  // rotary (cos, sin) in fp64: [total_frames][pt], then [frame_h][py], then [frame_w][px]
  const float2* rope32;   // the same table rounded to fp32
  int y_base, x_base;     // first row-axis and column-axis entries
  long long units_per_frame;  // T * h * d / 8
  int units_per_row;          // h * d / 8  (16-byte units per token)
  int units_per_head;         // d / 8
  int frame_w;
  int pt, py;                 // channel pairs on the time and row axes (pairs beyond pt+py: column axis)
  int px;
  int n_items;
  G1Item items[kMaxItems];
};

// ----------------------------------------------------------------- attention

// Attention work is described as query groups, each a run of query rows with
// its own list of key segments (row ranges of the K/V buffers).  A renderer or
// planner call is one group with one segment (the gathered context); a packed
// block-causal forward has one group per chunk with up to three segments
// (left anchor, right anchor, history + own chunk).
constexpr int kMaxGroups = 96;
constexpr int kMaxSegs = 3;

struct AttnGroup {
  int q_row0;              // first query row of the group
  int nq;                  // query rows
  int qb0;                 // first linear 256-row query block of the group
  int n_seg;               // key segments (1..kMaxSegs)
  int seg_row0[kMaxSegs];  // first key row of each segment
  int seg_rows[kMaxSegs];  // key rows of each segment
  int seg_tile0[kMaxSegs]; // first 128-key tile of each segment in the group's tile sequence
  int n_kv;                // tiles over all segments
};

struct AttnParams {
  void* out;            // bf16 [query rows, h, d]
  float* part_o;        // [pieces][256][d] unnormalised partial outputs (split only)
  float* part_ml;       // [pieces][256][2] running max (log2 units) and sum
  unsigned int* err;    // device error word
  int heads;
  int n_qb;             // linear 256-row query blocks over all groups
  int n_split;          // key-range splits per query block
  int n_pieces;         // heads * n_split * n_qb
  float scale_log2;     // log2(e) / sqrt(d)
  int n_groups;
  AttnGroup groups[kMaxGroups];
};

// Fill `p` with the single group [0, nq) x one key segment [0, nk).
inline void attn_single_group(AttnParams& p, int nq, int nk) {
  p.n_groups = 1;
  AttnGroup& g = p.groups[0];
  g.q_row0 = 0;
  g.nq = nq;
  g.qb0 = 0;
  g.n_seg = 1;
  g.seg_row0[0] = 0;
  g.seg_rows[0] = nk;
  g.seg_tile0[0] = 0;
  g.n_kv = (nk + 127) / 128;
  p.n_qb = (nq + 255) / 256;
}

// Host launchers (ff_publish.cu / ff_attn.cu).
cudaError_t launch_publish(const G1Params& p, int grid, cudaStream_t s);
cudaError_t launch_attention(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnParams& p, int grid, cudaStream_t s);
cudaError_t launch_combine(int head_dim, const AttnParams& p, cudaStream_t s);
size_t attention_smem_bytes(int head_dim);
cudaError_t launch_wait_probe(unsigned int* err, unsigned long long limit_ns, cudaStream_t s);
cudaError_t attention_configure(int head_dim);


}  // namespace ff
