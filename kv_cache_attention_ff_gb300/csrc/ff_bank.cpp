// Host side of libff: the bank state machine behind the C ABI in ff.h.
//
// State contract (FlashForward, onedev.kr/papers/332, "어떻게 동작하나", Eq. (2)):
// stage bank B_k of each layer holds H chunks; chunk i reads
// B_k^(i) = chunks max(0, i-H) .. i-1 and leaves B_k^(i+1) = Tail_H(B_k^(i) U (i, K, V)).
// Clean anchors (section "무엇과 다른가", stride Delta) live in a per-layer ring
// of anchor slots, anchor a in slot (a / Delta) mod cap.  Gamma(i): nearest
// anchor at or before the chunk's first frame and nearest at or after its last
// frame (dropped past the end; used once if both coincide).
//
// Storage: each (layer, stage) ring has H + 1 physical chunk slots, chunk j in
// physical slot j mod (H + 1), so chunk i is written into the slot of chunk
// i - H - 1, which no call reads any more, while chunks i - H .. i - 1 stay in
// place for its attention.  Logical slot j mod H (the contract's slot) maps to
// the physical slot of the resident chunk j.  K and V are separate planes
// ([ring slots][B_R frames] each, likewise [cap][1 frame] for anchors), so
// adjacent slots are adjacent rows and the attention reads the context as a
// few row runs in place (no gather copy).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "ff.h"
#include "ff_internal.h"

using namespace ff;

namespace {

bool log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FF_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

#define FF_LOG(...)                          \
  do {                                       \
    if (log_enabled()) {                     \
      std::fprintf(stderr, "[libff] " __VA_ARGS__); \
      std::fputc('\n', stderr);              \
    }                                        \
  } while (0)

struct SlotState {
  int tag = -1;
  int frames = 0;
};

// A run of adjacent slots read as one key segment: plane 0 = anchor slots of
// the layer, 1 = the (layer, stage) chunk ring, 2 = the planner's own-block
// scratch; `frames` counts frames from the first slot's start.
struct SegSpec {
  int plane;
  int slot;
  int frames;
};

struct TimedCall {
  cudaEvent_t ev[4];
  bool combine;
  int calls;     // renderer calls the events cover (a batch covers several)
  int launches;  // kernels launched between ev[0] and ev[3]
};

constexpr int kQBlock = 256;  // query rows per attention work unit
constexpr int kKTile = 128;   // keys per attention tile

}  // namespace

struct ff_bank {
  ff_bank_desc d{};
  int sm_count = 0;
  size_t frame_elems = 0;   // T * h * d
  size_t frame_bytes = 0;
  int max_key_frames = 0;
  int max_pieces = 0;
  size_t total_bytes = 0;
  std::vector<void*> allocations;

  int ring = 0;              // physical chunk slots per (layer, stage): H + 1

  // device memory
  uint8_t* stage_kv = nullptr;   // [L][S][K, V][H + 1 slots][B_R frames]
  uint8_t* q_rot_all = nullptr;  // [S][B_R frames]: every stage's rotated-Q scratch
  uint8_t* anchor_kv = nullptr;  // [L][K, V][cap][1 frame]
  struct Scratch {
    uint8_t* q_rot = nullptr;
    uint8_t* own_k = nullptr;    // planner: the block's rotated K, V
    uint8_t* own_v = nullptr;
    float* part_o = nullptr;
    float* part_ml = nullptr;
  };
  std::vector<Scratch> scratch;  // per stage
  Scratch planner;               // planner blocks (when planner_history > 0)
  int planner_max_pieces = 0;
  size_t part_rows = 0;          // capacity of each stage's split partials, in rows
  size_t planner_part_rows = 0;
  double2* rope64 = nullptr;
  float2* rope32 = nullptr;
  int rope_y_base = 0, rope_x_base = 0, pt = 0, py = 0, px = 0;
  unsigned int* err = nullptr;

  // host state
  std::vector<SlotState> stage_slots;   // [L][S][H + 1] physical slots
  std::vector<SlotState> anchor_slots;  // [L][cap]
  std::vector<int> next_chunk;          // [L][S]

  // cross-stream ordering
  std::vector<cudaEvent_t> ev_stage;       // [S] after the latest render of stage k
  std::vector<cudaStream_t> stage_stream;  // [S]
  std::vector<bool> stage_used;
  std::vector<cudaEvent_t> ev_anchor;      // [cap] after the latest publish touching the slot
  std::vector<cudaStream_t> anchor_stream;
  std::vector<bool> anchor_used;
  cudaEvent_t ev_planner = nullptr;        // after the latest planner call
  cudaStream_t planner_stream = nullptr;
  bool planner_used = false;

  // timing: a pool of event sets created by ff_bank_set_timing, reused by
  // later calls (the first n_timed are in use since the last reset)
  bool timing = false;
  std::vector<TimedCall> timed;
  size_t n_timed = 0;

  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;

  SlotState& sslot(int l, int s, int h) { return stage_slots[(static_cast<size_t>(l) * d.n_stages + s) * ring + h]; }
  const SlotState& sslot(int l, int s, int h) const {
    return stage_slots[(static_cast<size_t>(l) * d.n_stages + s) * ring + h];
  }
  SlotState& aslot(int l, int a) { return anchor_slots[static_cast<size_t>(l) * d.anchor_capacity + a]; }
  const SlotState& aslot(int l, int a) const { return anchor_slots[static_cast<size_t>(l) * d.anchor_capacity + a]; }

  size_t slot_bytes() const { return static_cast<size_t>(d.chunk_frames) * frame_bytes; }
  uint8_t* stage_k(int l, int s, int h) const {
    return stage_kv + (((static_cast<size_t>(l) * d.n_stages + s) * 2 + 0) * ring + h) * slot_bytes();
  }
  uint8_t* stage_v(int l, int s, int h) const {
    return stage_kv + (((static_cast<size_t>(l) * d.n_stages + s) * 2 + 1) * ring + h) * slot_bytes();
  }
  uint8_t* anchor_k(int l, int a) const {
    return anchor_kv + ((static_cast<size_t>(l) * 2 + 0) * d.anchor_capacity + a) * frame_bytes;
  }
  uint8_t* anchor_v(int l, int a) const {
    return anchor_kv + ((static_cast<size_t>(l) * 2 + 1) * d.anchor_capacity + a) * frame_bytes;
  }
};

namespace {

int n_chunks(const ff_bank_desc& d) { return (d.total_frames + d.chunk_frames - 1) / d.chunk_frames; }

int validate_desc(const ff_bank_desc* d) {
  if (!d) return FF_ERR_ARG;
  if (d->n_layers < 1 || d->n_stages < 1 || d->history < 1 || d->chunk_frames < 1 || d->chunk_frames > 8 ||
      d->anchor_stride < 1 || d->anchor_capacity < 1 || d->total_frames < 1 || d->heads < 1 ||
      (d->head_dim != 64 && d->head_dim != 128) || d->frame_h < 1 || d->frame_w < 1 || !(d->rope_theta > 0.0) ||
      d->device < 0)
    return FF_ERR_ARG;
  if (2 + (d->history + 1) * d->chunk_frames > kMaxItems) return FF_ERR_ARG;
  if (d->planner_block < 1 || d->planner_block > 8 || d->planner_history < 0 ||
      (d->planner_history + 1) * d->planner_block > kMaxItems)
    return FF_ERR_ARG;
  const long long T = static_cast<long long>(d->frame_h) * d->frame_w;
  const long long upf = T * d->heads * d->head_dim / 8;
  // every count the kernels index with 32-bit ints must fit
  if (upf * (2 + (d->history + 1) * d->chunk_frames) > (1ll << 31) - 1) return FF_ERR_ARG;
  if (T * (2 + (d->history + 1) * d->chunk_frames) > (1ll << 30)) return FF_ERR_ARG;
  if (upf * (d->planner_history + 1) * d->planner_block > (1ll << 31) - 1) return FF_ERR_ARG;
  if (static_cast<long long>(d->heads) * d->head_dim * 2 % 16 != 0) return FF_ERR_ARG;
  if (upf >= (1ll << 24)) return FF_ERR_ARG;  // the publish kernel's index math is exact below 2^24 units
  return FF_OK;
}

void plan(const ff_bank_desc& d, int i, ff_chunk_plan* p) {
  const int s = d.chunk_frames * i;
  const int e = std::min(s + d.chunk_frames - 1, d.total_frames - 1);
  p->first_frame = s;
  p->n_frames = e - s + 1;
  const int left = d.anchor_stride * (s / d.anchor_stride);
  const int right = d.anchor_stride * ((e + d.anchor_stride - 1) / d.anchor_stride);
  p->anchors[0] = left;
  p->anchors[1] = -1;
  p->n_anchors = 1;
  if (right != left && right <= d.total_frames - 1) {
    p->anchors[1] = right;
    p->n_anchors = 2;
  }
  p->hist_first = std::max(0, i - d.history);
  p->n_hist = i - p->hist_first;
  int hf = 0;
  for (int j = p->hist_first; j < i; ++j) {
    const int js = d.chunk_frames * j;
    hf += std::min(js + d.chunk_frames - 1, d.total_frames - 1) - js + 1;
  }
  p->hist_frames = hf;
  p->slot = i % d.history;
  p->key_frames = p->n_anchors + hf + p->n_frames;
}

int n_anchor_frames(const ff_bank_desc& d) { return (d.total_frames - 1) / d.anchor_stride + 1; }
int n_planner_blocks(const ff_bank_desc& d) { return (n_anchor_frames(d) + d.planner_block - 1) / d.planner_block; }

// Planner block b: anchors b*B_P .. b*B_P + n - 1; history = the anchors of blocks
// max(0, b - H_P) .. b - 1, all full blocks.
void plan_planner(const ff_bank_desc& d, int b, ff_planner_plan* p) {
  p->first_anchor = b * d.planner_block;
  p->n_anchors = std::min(d.planner_block, n_anchor_frames(d) - p->first_anchor);
  p->hist_first_block = std::max(0, b - d.planner_history);
  p->n_hist_blocks = b - p->hist_first_block;
  p->hist_frames = p->n_hist_blocks * d.planner_block;
  p->key_frames = p->hist_frames + p->n_anchors;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_err(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FF_OK;
  FF_LOG("%s: %s", what, cudaGetErrorString(e));
  return FF_ERR_CUDA;
}

// 2-D tensor map over a bf16 [rows, heads * head_dim] buffer, 64 x 128 boxes, 128-byte swizzle.
int make_map(const ff_bank* b, CUtensorMap* map, const void* base, int rows, int box_rows = 128) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(b->d.heads) * b->d.head_dim, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(b->d.heads) * b->d.head_dim * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = b->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    FF_LOG("cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return FF_ERR_CUDA;
  }
  return FF_OK;
}

// Append anchor slot `sl` (one frame) to `seg`, extending the last run when
// the slot is physically next to it.
void add_anchor_slot(std::vector<SegSpec>& seg, int sl) {
  if (!seg.empty() && seg.back().plane == 0 && seg.back().slot + seg.back().frames == sl)
    ++seg.back().frames;
  else
    seg.push_back({0, sl, 1});
}

// Key segments of chunk i: runs of adjacent anchor slots of Gamma(i), then runs
// of adjacent ring slots holding chunks max(0, i-H) .. i (chunk j in physical
// slot j mod (H+1)); a run continues past a slot only when that slot is full.
std::vector<SegSpec> chunk_segments(const ff_bank_desc& d, int chunk, const ff_chunk_plan& pl) {
  std::vector<SegSpec> seg;
  for (int j = 0; j < pl.n_anchors; ++j) add_anchor_slot(seg, (pl.anchors[j] / d.anchor_stride) % d.anchor_capacity);
  const int ring = d.history + 1;
  std::vector<int> fr(ring, 0);
  for (int j = pl.hist_first; j <= chunk; ++j) {
    const int js = d.chunk_frames * j;
    fr[j % ring] = std::min(js + d.chunk_frames - 1, d.total_frames - 1) - js + 1;
  }
  for (int h = 0; h < ring; ++h) {
    if (!fr[h]) continue;
    if (h > 0 && fr[h - 1] == d.chunk_frames && !seg.empty() && seg.back().plane == 1)
      seg.back().frames += fr[h];
    else
      seg.push_back({1, h, fr[h]});
  }
  return seg;
}

// Key segments of planner block b: runs of the history blocks' anchor slots,
// then the block's own rotated K/V (scratch).
std::vector<SegSpec> planner_segments(const ff_bank_desc& d, const ff_planner_plan& pl) {
  std::vector<SegSpec> seg;
  for (int j = 0; j < pl.hist_frames; ++j)
    add_anchor_slot(seg, (pl.hist_first_block * d.planner_block + j) % d.anchor_capacity);
  seg.push_back({2, 0, pl.n_anchors});
  return seg;
}

int tiles_of(const std::vector<SegSpec>& seg, long long T) {
  int tiles = 0;
  for (const SegSpec& g : seg) tiles += static_cast<int>((g.frames * T + kKTile - 1) / kKTile);
  return tiles;
}

// Fill group `g`'s key segments and the launch's K/V maps m0, m0 + 1, ...
// (one pair per segment, each ending where its segment ends).  `base` gives
// each segment's first K and V frame.
template <class Base, class KV>
int build_segments(const ff_bank* b, const std::vector<SegSpec>& seg, Base base, AttnGroup& g, KV& kv, int m0 = 0) {
  if (seg.empty() || seg.size() > static_cast<size_t>(kMaxSegs) || m0 + static_cast<int>(seg.size()) > KV::kMaps)
    return FF_ERR_ARG;
  const long long T = static_cast<long long>(b->d.frame_h) * b->d.frame_w;
  g.n_seg = 0;
  int tiles = 0;
  for (const SegSpec& sp : seg) {
    const void* k = nullptr;
    const void* v = nullptr;
    base(sp, &k, &v);
    const long long rows = sp.frames * T;
    const int m = m0 + g.n_seg;
    int rc;
    if ((rc = make_map(b, &kv.k[m], k, static_cast<int>(rows))) != FF_OK) return rc;
    if ((rc = make_map(b, &kv.v[m], v, static_cast<int>(rows))) != FF_OK) return rc;
    g.seg_map[g.n_seg] = m;
    g.seg_row0[g.n_seg] = 0;
    g.seg_rows[g.n_seg] = static_cast<int>(rows);
    g.seg_tile0[g.n_seg] = tiles;
    tiles += static_cast<int>((rows + kKTile - 1) / kKTile);
    ++g.n_seg;
  }
  g.n_kv = tiles;
  return FF_OK;
}

// Unused map entries of a launch stay valid descriptors (copies of entry 0,
// which every launch uses): entries [used, kMaps), or those not marked in `used`.
template <class KV>
void fill_unused_maps(KV& kv, int used) {
  for (int m = used; m < KV::kMaps; ++m) {
    kv.k[m] = kv.k[0];
    kv.v[m] = kv.v[0];
  }
}
template <class KV>
void fill_unused_maps(KV& kv, const bool* used) {
  for (int m = 1; m < KV::kMaps; ++m)
    if (!used[m]) {
      kv.k[m] = kv.k[0];
      kv.v[m] = kv.v[0];
    }
}

// Work plan and Q tensor map of an attention launch for the query groups in
// `ap` (heads, out, err, scale and groups filled by the caller): everything
// that can fail before a kernel is enqueued.  Partial rows beyond `part_rows`
// disable splitting.
int prepare_attention(const ff_bank* b, AttnParams& ap, const void* q, int q_rows, float* part_o, float* part_ml,
                      size_t part_rows, bool allow_split, CUtensorMap* tq) {
  ap.part_o = part_o;
  ap.part_ml = part_ml;
  const int rc = make_map(b, tq, q, q_rows);
  if (rc != FF_OK) return rc;
  const int units = b->d.heads * ap.n_qb;
  SplitPlan sp{units, 1, units, 0};
  // the planner's cost model assumes one key-tile count for every unit
  bool uniform = true;
  for (int g = 1; g < ap.n_groups; ++g) uniform = uniform && ap.groups[g].n_kv == ap.groups[0].n_kv;
  if (allow_split && uniform) sp = plan_split(units, ap.groups[0].n_kv, b->sm_count, part_rows);
  ap.n_whole = sp.n_whole;
  ap.n_split = sp.n_split;
  ap.n_pieces = sp.n_pieces;
  return FF_OK;
}

// Launch attention (and the split combine) prepared by prepare_attention over
// the K/V maps `kv`.  With `tc`, ev[2] is recorded between attention and combine.
template <class KV>
int attend(const ff_bank* b, const AttnParams& ap, const CUtensorMap& tq, const KV& kv, cudaStream_t s,
           TimedCall* tc) {
  int rc;
  const int grid = std::min(ap.n_pieces, b->sm_count);
  if ((rc = cuda_err(launch_attention(b->d.head_dim, tq, kv, ap, grid, s), "attention launch")) != FF_OK) return rc;
  if (tc) cudaEventRecord(tc->ev[2], s);
  if (ap.n_split > 1 && (rc = cuda_err(launch_combine(b->d.head_dim, ap, s), "combine launch")) != FF_OK) return rc;
  if (tc) {
    tc->combine = ap.n_split > 1;
    tc->launches += ap.n_split > 1 ? 2 : 1;
  }
  return FF_OK;
}

// Common fields of a RoPE/publish launch.
G1Params publish_params(const ff_bank* b) {
  const ff_bank_desc& d = b->d;
  G1Params prm{};
  prm.rope64 = b->rope64;
  prm.rope32 = b->rope32;
  prm.y_base = b->rope_y_base;
  prm.x_base = b->rope_x_base;
  prm.units_per_frame = static_cast<long long>(b->frame_elems / 8);
  prm.units_per_row = d.heads * d.head_dim / 8;
  prm.units_per_head = d.head_dim / 8;
  prm.frame_w = d.frame_w;
  prm.inv_frame_w = static_cast<float>(1.0 / d.frame_w);
  prm.pt = b->pt;
  prm.py = b->py;
  prm.px = b->px;
  return prm;
}

G1Item rot_item(const void* src_k, const void* src_v, void* dst_k, void* dst_v, int t, const void* src_q = nullptr,
                void* dst_q = nullptr) {
  G1Item it{};
  it.src_k = src_k;
  it.src_v = src_v;
  it.src_q = src_q;
  it.dst_k = dst_k;
  it.dst_v = dst_v;
  it.dst_q = dst_q;
  it.t = t;
  return it;
}

const uint8_t* frame_at(const void* base, size_t frame, size_t frame_bytes) {
  return static_cast<const uint8_t*>(base) + frame * frame_bytes;
}

void free_all(ff_bank* b) {
  for (void* p : b->allocations) cudaFree(p);
  b->allocations.clear();
  for (cudaEvent_t e : b->ev_stage)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : b->ev_anchor)
    if (e) cudaEventDestroy(e);
  for (auto& tc : b->timed)
    for (cudaEvent_t e : tc.ev) cudaEventDestroy(e);
  if (b->ev_planner) cudaEventDestroy(b->ev_planner);
  b->ev_planner = nullptr;
  b->ev_stage.clear();
  b->ev_anchor.clear();
  b->timed.clear();
}

int alloc(ff_bank* b, size_t bytes, void** out) {
  if (bytes == 0) bytes = 16;
  void* p = nullptr;
  const cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    FF_LOG("cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    return FF_ERR_OOM;
  }
  b->allocations.push_back(p);
  *out = p;
  return FF_OK;
}

// Timing event sets: kTimedPool are created when timing is switched on, so a
// timed render records into existing events; a run with more calls between
// resets grows the pool by that many again.
constexpr size_t kTimedPool = 2048;

int grow_timed(ff_bank* b, size_t n) {
  for (size_t j = 0; j < n; ++j) {
    TimedCall tc{};
    for (auto& e : tc.ev)
      if (cudaEventCreate(&e) != cudaSuccess) {
        for (auto& f : tc.ev)
          if (f) cudaEventDestroy(f);
        return FF_ERR_CUDA;
      }
    b->timed.push_back(tc);
  }
  return FF_OK;
}

int next_timed_call(ff_bank* b, TimedCall** tc) {
  if (b->n_timed == b->timed.size()) {
    const int rc = grow_timed(b, kTimedPool);
    if (rc != FF_OK) return rc;
  }
  *tc = &b->timed[b->n_timed];
  (*tc)->combine = false;
  (*tc)->calls = 1;
  (*tc)->launches = 0;
  return FF_OK;
}

// Make `s` wait for the last render of every stage that ran on another stream.
void wait_stage_events(ff_bank* b, cudaStream_t s, int only_stage) {
  for (int k = 0; k < b->d.n_stages; ++k) {
    if (only_stage >= 0 && k != only_stage) continue;
    if (b->stage_used[k] && b->stage_stream[k] != s) cudaStreamWaitEvent(s, b->ev_stage[k], 0);
  }
}

// One renderer call, checked and planned: everything about it that can fail
// is found here, before any work is enqueued.
struct RenderCall {
  ff_render_call c;
  ff_chunk_plan pl;
  int aslots[2];
  int own_phys;
  std::vector<SegSpec> seg;
};

int check_render_call(const ff_bank* b, const ff_render_call& c, RenderCall* rc) {
  const ff_bank_desc& d = b->d;
  if (c.layer < 0 || c.layer >= d.n_layers || c.stage < 0 || c.stage >= d.n_stages || c.chunk < 0 ||
      c.chunk >= n_chunks(d) || !c.q_pre || !c.k_pre || !c.v || !c.out || !aligned16(c.q_pre) || !aligned16(c.k_pre) ||
      !aligned16(c.v) || !aligned16(c.out))
    return FF_ERR_ARG;
  if (c.chunk != b->next_chunk[static_cast<size_t>(c.layer) * d.n_stages + c.stage]) return FF_ERR_ORDER;
  rc->c = c;
  plan(d, c.chunk, &rc->pl);
  const ff_chunk_plan& pl = rc->pl;
  for (int j = 0; j < pl.n_anchors; ++j) {
    rc->aslots[j] = (pl.anchors[j] / d.anchor_stride) % d.anchor_capacity;
    if (b->aslot(c.layer, rc->aslots[j]).tag != pl.anchors[j]) return FF_ERR_ANCHOR_MISSING;
  }
  rc->own_phys = c.chunk % b->ring;
  for (int jc = pl.hist_first; jc < c.chunk; ++jc)
    if (b->sslot(c.layer, c.stage, jc % b->ring).tag != jc) return FF_ERR_ARG;  // internal invariant (Tail_H) broken
  rc->seg = chunk_segments(d, c.chunk, pl);
  int key_frames = 0;
  for (const SegSpec& g : rc->seg) key_frames += g.frames;
  return key_frames == pl.key_frames ? FF_OK : FF_ERR_ARG;
}

// The call's publish items: RoPE of its Q frames into `q_rot`, RoPE(K) and V
// into its ring slot.
void add_render_items(const ff_bank* b, const RenderCall& r, uint8_t* q_rot, G1Params& prm) {
  const ff_render_call& c = r.c;
  for (int f = 0; f < r.pl.n_frames; ++f)
    prm.items[prm.n_items++] =
        rot_item(frame_at(c.k_pre, f, b->frame_bytes), frame_at(c.v, f, b->frame_bytes),
                 b->stage_k(c.layer, c.stage, r.own_phys) + static_cast<size_t>(f) * b->frame_bytes,
                 b->stage_v(c.layer, c.stage, r.own_phys) + static_cast<size_t>(f) * b->frame_bytes,
                 r.pl.first_frame + f, frame_at(c.q_pre, f, b->frame_bytes), q_rot + static_cast<size_t>(f) * b->frame_bytes);
}

// The call's query group: rows q_row0 .. of the launch's Q map, key segments
// read in place through maps m0, m0 + 1, ...
template <class KV>
int add_render_group(const ff_bank* b, const RenderCall& r, int q_row0, int qb0, AttnGroup& g, KV& kv, int m0) {
  const ff_render_call& c = r.c;
  const long long T = static_cast<long long>(b->d.frame_h) * b->d.frame_w;
  g.q_row0 = q_row0;
  g.nq = static_cast<int>(r.pl.n_frames * T);
  g.qb0 = qb0;
  g.out = c.out;
  g.out_row0 = 0;
  return build_segments(b, r.seg,
                        [&](const SegSpec& sg, const void** k, const void** vv) {
                          *k = sg.plane == 0 ? b->anchor_k(c.layer, sg.slot) : b->stage_k(c.layer, c.stage, sg.slot);
                          *vv = sg.plane == 0 ? b->anchor_v(c.layer, sg.slot) : b->stage_v(c.layer, c.stage, sg.slot);
                        },
                        g, kv, m0);
}

// Bank state after a call: its chunk is resident in its ring slot.
void commit_render(ff_bank* b, const RenderCall& r) {
  SlotState& own = b->sslot(r.c.layer, r.c.stage, r.own_phys);
  own.tag = r.c.chunk;
  own.frames = r.pl.n_frames;
  ++b->next_chunk[static_cast<size_t>(r.c.layer) * b->d.n_stages + r.c.stage];
}

// n independent renderer calls (distinct stages when n > 1) as one RoPE/publish
// launch and one attention launch (plus the split combine when planned).  Every
// check runs before the first launch.
int render_calls(ff_bank* b, int n, const ff_render_call* calls, cudaStream_t s) {
  const ff_bank_desc& d = b->d;
  RenderCall rcs[kMaxBatch];
  int rc;
  for (int j = 0; j < n; ++j) {
    for (int i = 0; i < j; ++i)
      if (calls[i].stage == calls[j].stage) return FF_ERR_ARG;  // one call per stage bank and scratch
    if ((rc = check_render_call(b, calls[j], &rcs[j])) != FF_OK) return rc;
  }
  if (cudaSetDevice(d.device) != cudaSuccess) return FF_ERR_CUDA;
  const long long T = static_cast<long long>(d.frame_h) * d.frame_w;
  const int slot_rows = static_cast<int>(d.chunk_frames * T);  // Q rows of one stage's scratch

  G1Params prm = publish_params(b);
  prm.n_items = 0;
  AttnParams ap{};
  ap.err = b->err;
  ap.heads = d.heads;
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.head_dim)));
  ap.n_groups = n;
  KVMaps kv1;
  KVMapsBatch kvb;
  int qb = 0;
  for (int j = 0; j < n; ++j) {
    const RenderCall& r = rcs[j];
    add_render_items(b, r, b->scratch[r.c.stage].q_rot, prm);
    // every stage's Q scratch is a row range of one buffer: one Q map serves the batch
    const int q_row0 = n == 1 ? 0 : r.c.stage * slot_rows;
    rc = n == 1 ? add_render_group(b, r, q_row0, qb, ap.groups[j], kv1, 0)
                : add_render_group(b, r, q_row0, qb, ap.groups[j], kvb, j * kMaxMaps);
    if (rc != FF_OK) return rc;
    qb += (ap.groups[j].nq + kQBlock - 1) / kQBlock;
  }
  ap.n_qb = qb;
  if (n == 1) {
    fill_unused_maps(kv1, static_cast<int>(rcs[0].seg.size()));
  } else {
    bool used[KVMapsBatch::kMaps] = {};
    for (int j = 0; j < n; ++j)
      for (size_t m = 0; m < rcs[j].seg.size(); ++m) used[j * kMaxMaps + m] = true;
    fill_unused_maps(kvb, used);
  }
  // the first call's stage scratch holds the split partials of the launch
  ff_bank::Scratch& sc = b->scratch[rcs[0].c.stage];
  const void* q_map_base = n == 1 ? static_cast<const void*>(sc.q_rot) : static_cast<const void*>(b->q_rot_all);
  const int q_map_rows = n == 1 ? rcs[0].pl.n_frames * static_cast<int>(T) : d.n_stages * slot_rows;
  CUtensorMap tq;
  if ((rc = prepare_attention(b, ap, q_map_base, q_map_rows, sc.part_o, sc.part_ml, b->part_rows, true, &tq)) != FF_OK)
    return rc;
  TimedCall* tc = nullptr;
  if (b->timing && (rc = next_timed_call(b, &tc)) != FF_OK) return rc;

  // ---- ordering against other streams
  for (int j = 0; j < n; ++j) {
    const RenderCall& r = rcs[j];
    wait_stage_events(b, s, r.c.stage);
    for (int a = 0; a < r.pl.n_anchors; ++a)
      if (b->anchor_used[r.aslots[a]] && b->anchor_stream[r.aslots[a]] != s)
        cudaStreamWaitEvent(s, b->ev_anchor[r.aslots[a]], 0);
  }

  // ---- nothing below fails for a reason that can be checked beforehand
  if (tc) {
    tc->calls = n;
    tc->launches = 1;
    cudaEventRecord(tc->ev[0], s);
  }
  if ((rc = cuda_err(launch_publish(prm, 0, s), "publish launch")) != FF_OK) return rc;
  if (tc) cudaEventRecord(tc->ev[1], s);
  rc = n == 1 ? attend(b, ap, tq, kv1, s, tc) : attend(b, ap, tq, kvb, s, tc);
  if (rc != FF_OK) return rc;
  if (tc) {
    cudaEventRecord(tc->ev[3], s);
    ++b->n_timed;
  }
  for (int j = 0; j < n; ++j) {
    const int st = rcs[j].c.stage;
    cudaEventRecord(b->ev_stage[st], s);
    b->stage_stream[st] = s;
    b->stage_used[st] = true;
    commit_render(b, rcs[j]);
  }
  return FF_OK;
}

}  // namespace

extern "C" {

int ff_desc_default(ff_bank_desc* d) {
  if (!d) return FF_ERR_ARG;
  std::memset(d, 0, sizeof(*d));
  d->n_layers = 1;
  d->n_stages = 4;
  d->history = 5;
  d->chunk_frames = 3;
  d->anchor_stride = 10;
  d->anchor_capacity = 9;
  d->total_frames = 81;
  d->heads = 12;
  d->head_dim = 128;
  d->frame_h = 30;
  d->frame_w = 52;
  d->rope_theta = 10000.0;
  d->max_bytes = 0;
  d->device = 0;
  d->planner_block = 3;
  d->planner_history = 6;
  return FF_OK;
}

const char* ff_status_string(int s) {
  switch (s) {
    case FF_OK: return "ok";
    case FF_ERR_ARG: return "invalid argument";
    case FF_ERR_ORDER: return "chunk out of order for this (layer, stage)";
    case FF_ERR_ANCHOR_MISSING: return "anchor of Gamma(i) not resident";
    case FF_ERR_OOM: return "out of device memory (or over max_bytes)";
    case FF_ERR_CUDA: return "CUDA runtime error";
    case FF_ERR_DEVICE_TIMEOUT: return "bounded device wait timed out";
    case FF_ERR_UNSUPPORTED: return "device is not sm_103";
    default: return "unknown status";
  }
}

int ff_plan_chunk(const ff_bank_desc* d, int chunk, ff_chunk_plan* out) {
  if (validate_desc(d) != FF_OK || !out || chunk < 0 || chunk >= n_chunks(*d)) return FF_ERR_ARG;
  plan(*d, chunk, out);
  return FF_OK;
}

int ff_bank_create(const ff_bank_desc* desc, ff_bank_t** out) {
  if (!out) return FF_ERR_ARG;
  const int v = validate_desc(desc);
  if (v != FF_OK) return v;
  const ff_bank_desc& d = *desc;

  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) != cudaSuccess || d.device >= dev_count) {
    cudaGetLastError();
    return FF_ERR_CUDA;
  }
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, d.device) != cudaSuccess) return FF_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return FF_ERR_UNSUPPORTED;
  if (cudaSetDevice(d.device) != cudaSuccess) return FF_ERR_CUDA;

  ff_bank* b = new ff_bank();
  b->d = d;
  b->sm_count = prop.multiProcessorCount;
  const size_t T = static_cast<size_t>(d.frame_h) * d.frame_w;
  b->frame_elems = T * d.heads * d.head_dim;
  b->frame_bytes = b->frame_elems * 2;
  b->max_key_frames = 2 + (d.history + 1) * d.chunk_frames;
  b->ring = d.history + 1;

  // attention split scratch: the most partial rows any call of this bank can
  // use (a call's key tiles exceed ceil(keys / 128) by at most kMaxSegs - 1)
  auto rows_cap = [&](int q_frames, int k_frames) {
    size_t m = 0;
    for (int f = 1; f <= q_frames; ++f) {
      const int nq = static_cast<int>(f * T);
      const int n_qb = (nq + kQBlock - 1) / kQBlock;
      for (int kf = f; kf <= k_frames; ++kf)
        for (int extra = 0; extra < kMaxSegs; ++extra) {
          const int n_kv = static_cast<int>((kf * T + kKTile - 1) / kKTile) + extra;
          m = std::max(m, plan_split(d.heads * n_qb, n_kv, b->sm_count, static_cast<size_t>(-1)).part_rows);
        }
    }
    return m;
  };
  b->part_rows = rows_cap(d.chunk_frames, b->max_key_frames);
  const int planner_frames = (d.planner_history + 1) * d.planner_block;
  b->planner_part_rows = d.planner_history > 0 ? rows_cap(d.planner_block, planner_frames) : 0;
  const int max_pieces = static_cast<int>(b->part_rows / kQBlock);
  b->max_pieces = max_pieces;
  b->planner_max_pieces = static_cast<int>(b->planner_part_rows / kQBlock);

  const int pt = (d.head_dim - 4 * (d.head_dim / 6)) / 2;
  const int py = (d.head_dim / 6);
  const int px = (d.head_dim / 6);
  b->pt = pt;
  b->py = py;
  b->px = px;
  b->rope_y_base = d.total_frames * pt;
  b->rope_x_base = b->rope_y_base + d.frame_h * py;
  const size_t n_rope = static_cast<size_t>(b->rope_x_base) + static_cast<size_t>(d.frame_w) * px;

  const size_t stage_bytes = static_cast<size_t>(d.n_layers) * d.n_stages * b->ring * 2 * b->slot_bytes();
  const size_t anchor_bytes = static_cast<size_t>(d.n_layers) * d.anchor_capacity * 2 * b->frame_bytes;
  const size_t qrot_bytes = b->slot_bytes();
  const size_t part_o_bytes = static_cast<size_t>(max_pieces) * kQBlock * d.head_dim * 4;
  const size_t part_ml_bytes = static_cast<size_t>(max_pieces) * kQBlock * 8;
  const size_t per_stage = qrot_bytes + part_o_bytes + part_ml_bytes;
  const size_t rope_bytes = n_rope * (sizeof(double2) + sizeof(float2));
  const size_t pl_block_bytes = static_cast<size_t>(d.planner_block) * b->frame_bytes;
  const size_t pl_part_o_bytes = static_cast<size_t>(b->planner_max_pieces) * kQBlock * d.head_dim * 4;
  const size_t pl_part_ml_bytes = static_cast<size_t>(b->planner_max_pieces) * kQBlock * 8;
  const size_t planner_bytes = d.planner_history > 0 ? 3 * pl_block_bytes + pl_part_o_bytes + pl_part_ml_bytes : 0;
  b->total_bytes = stage_bytes + anchor_bytes + d.n_stages * per_stage + planner_bytes + rope_bytes + 256;
  if (d.max_bytes && b->total_bytes > d.max_bytes) {
    FF_LOG("bank needs %zu bytes > max_bytes %zu", b->total_bytes, d.max_bytes);
    delete b;
    return FF_ERR_OOM;
  }

  int rc = FF_OK;
  void* p = nullptr;
  if ((rc = alloc(b, stage_bytes, &p)) != FF_OK) goto fail;
  b->stage_kv = static_cast<uint8_t*>(p);
  if ((rc = alloc(b, anchor_bytes, &p)) != FF_OK) goto fail;
  b->anchor_kv = static_cast<uint8_t*>(p);
  b->scratch.resize(d.n_stages);
  if ((rc = alloc(b, qrot_bytes * d.n_stages, &p)) != FF_OK) goto fail;
  b->q_rot_all = static_cast<uint8_t*>(p);
  for (int k = 0; k < d.n_stages; ++k) {
    b->scratch[k].q_rot = b->q_rot_all + static_cast<size_t>(k) * qrot_bytes;
    if ((rc = alloc(b, part_o_bytes, &p)) != FF_OK) goto fail;
    b->scratch[k].part_o = static_cast<float*>(p);
    if ((rc = alloc(b, part_ml_bytes, &p)) != FF_OK) goto fail;
    b->scratch[k].part_ml = static_cast<float*>(p);
  }
  if (d.planner_history > 0) {
    if ((rc = alloc(b, pl_block_bytes, &p)) != FF_OK) goto fail;
    b->planner.own_k = static_cast<uint8_t*>(p);
    if ((rc = alloc(b, pl_block_bytes, &p)) != FF_OK) goto fail;
    b->planner.own_v = static_cast<uint8_t*>(p);
    if ((rc = alloc(b, pl_block_bytes, &p)) != FF_OK) goto fail;
    b->planner.q_rot = static_cast<uint8_t*>(p);
    if ((rc = alloc(b, pl_part_o_bytes, &p)) != FF_OK) goto fail;
    b->planner.part_o = static_cast<float*>(p);
    if ((rc = alloc(b, pl_part_ml_bytes, &p)) != FF_OK) goto fail;
    b->planner.part_ml = static_cast<float*>(p);
  }
  if ((rc = alloc(b, n_rope * sizeof(double2), &p)) != FF_OK) goto fail;
  b->rope64 = static_cast<double2*>(p);
  if ((rc = alloc(b, n_rope * sizeof(float2), &p)) != FF_OK) goto fail;
  b->rope32 = static_cast<float2*>(p);
  if ((rc = alloc(b, 256, &p)) != FF_OK) goto fail;
  b->err = static_cast<unsigned int*>(p);

  {
    // Rotary table: omega_j = theta^(-2j / d_axis), angle = position * omega_j (fp64), libm cos/sin.
    std::vector<double2> h64(n_rope);
    std::vector<float2> h32(n_rope);
    auto fill = [&](size_t base, int n_pos, int pairs, int d_axis) {
      for (int pos = 0; pos < n_pos; ++pos)
        for (int j = 0; j < pairs; ++j) {
          const double omega = std::pow(d.rope_theta, -static_cast<double>(2 * j) / static_cast<double>(d_axis));
          const double ang = static_cast<double>(pos) * omega;
          const double c = std::cos(ang), s = std::sin(ang);
          h64[base + static_cast<size_t>(pos) * pairs + j] = make_double2(c, s);
          h32[base + static_cast<size_t>(pos) * pairs + j] = make_float2(static_cast<float>(c), static_cast<float>(s));
        }
    };
    fill(0, d.total_frames, pt, 2 * pt);
    fill(b->rope_y_base, d.frame_h, py, 2 * py);
    fill(b->rope_x_base, d.frame_w, px, 2 * px);
    if (cudaMemcpy(b->rope64, h64.data(), n_rope * sizeof(double2), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(b->rope32, h32.data(), n_rope * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(b->err, 0, 256) != cudaSuccess) {
      rc = FF_ERR_CUDA;
      goto fail;
    }
  }
  {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
      rc = FF_ERR_CUDA;
      goto fail;
    }
    b->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (attention_configure(d.head_dim) != cudaSuccess) {
    rc = FF_ERR_CUDA;
    goto fail;
  }

  b->stage_slots.assign(static_cast<size_t>(d.n_layers) * d.n_stages * b->ring, SlotState{});
  b->anchor_slots.assign(static_cast<size_t>(d.n_layers) * d.anchor_capacity, SlotState{});
  b->next_chunk.assign(static_cast<size_t>(d.n_layers) * d.n_stages, 0);
  b->ev_stage.assign(d.n_stages, nullptr);
  b->stage_stream.assign(d.n_stages, nullptr);
  b->stage_used.assign(d.n_stages, false);
  b->ev_anchor.assign(d.anchor_capacity, nullptr);
  b->anchor_stream.assign(d.anchor_capacity, nullptr);
  b->anchor_used.assign(d.anchor_capacity, false);
  for (auto& e : b->ev_stage)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      rc = FF_ERR_CUDA;
      goto fail;
    }
  for (auto& e : b->ev_anchor)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      rc = FF_ERR_CUDA;
      goto fail;
    }
  if (cudaEventCreateWithFlags(&b->ev_planner, cudaEventDisableTiming) != cudaSuccess) {
    rc = FF_ERR_CUDA;
    goto fail;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    rc = FF_ERR_CUDA;
    goto fail;
  }
  FF_LOG("bank created: %zu bytes, %d SMs, max pieces %d", b->total_bytes, b->sm_count, max_pieces);
  *out = b;
  return FF_OK;

fail:
  free_all(b);
  delete b;
  return rc;
}

int ff_bank_destroy(ff_bank_t* b) {
  if (!b) return FF_OK;
  cudaSetDevice(b->d.device);
  cudaDeviceSynchronize();
  free_all(b);
  delete b;
  return FF_OK;
}

int ff_bank_gamma(const ff_bank_t* b, int chunk, int* left, int* right, int* n) {
  if (!b || chunk < 0 || chunk >= n_chunks(b->d)) return FF_ERR_ARG;
  ff_chunk_plan p;
  plan(b->d, chunk, &p);
  if (left) *left = p.anchors[0];
  if (right) *right = p.anchors[1];
  if (n) *n = p.n_anchors;
  return FF_OK;
}

int ff_bank_slot_info(const ff_bank_t* b, int layer, int stage, int slot, int* chunk_tag, int* frames,
                      const void** k, const void** v) {
  if (!b || layer < 0 || layer >= b->d.n_layers || stage < -1 || stage >= b->d.n_stages) return FF_ERR_ARG;
  if (stage == -1) {
    if (slot < 0 || slot >= b->d.anchor_capacity) return FF_ERR_ARG;
    const SlotState& s = b->aslot(layer, slot);
    if (chunk_tag) *chunk_tag = s.tag;
    if (frames) *frames = s.frames;
    if (k) *k = b->anchor_k(layer, slot);
    if (v) *v = b->anchor_v(layer, slot);
    return FF_OK;
  }
  if (slot < 0 || slot >= b->d.history) return FF_ERR_ARG;
  // logical slot `slot` holds the resident chunk j (of the last H) with j mod H == slot
  const int next = b->next_chunk[static_cast<size_t>(layer) * b->d.n_stages + stage];
  int phys = slot, tag = -1, fr = 0;
  for (int j = std::max(0, next - b->d.history); j < next; ++j)
    if (j % b->d.history == slot) {
      phys = j % b->ring;
      const SlotState& s = b->sslot(layer, stage, phys);
      tag = s.tag;
      fr = s.frames;
    }
  if (chunk_tag) *chunk_tag = tag;
  if (frames) *frames = fr;
  if (k) *k = b->stage_k(layer, stage, phys);
  if (v) *v = b->stage_v(layer, stage, phys);
  return FF_OK;
}

int ff_bank_bytes(const ff_bank_t* b, size_t* bytes) {
  if (!b || !bytes) return FF_ERR_ARG;
  *bytes = b->total_bytes;
  return FF_OK;
}

int ff_bank_error_poll(ff_bank_t* b) {
  if (!b) return FF_ERR_ARG;
  cudaSetDevice(b->d.device);
  if (cudaDeviceSynchronize() != cudaSuccess) return FF_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, b->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FF_ERR_CUDA;
  if (word) {
    cudaMemset(b->err, 0, sizeof(word));
    return FF_ERR_DEVICE_TIMEOUT;
  }
  return FF_OK;
}

int ff_anchor_publish(ff_bank_t* b, int layer, int first, int n, const void* k_pre, const void* v, void* stream) {
  if (!b || layer < 0 || layer >= b->d.n_layers || n < 1 || n > b->d.anchor_capacity || n > kMaxItems || first < 0 ||
      first % b->d.anchor_stride != 0 || first + (n - 1) * b->d.anchor_stride > b->d.total_frames - 1 || !k_pre ||
      !v || !aligned16(k_pre) || !aligned16(v))
    return FF_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaSetDevice(b->d.device) != cudaSuccess) return FF_ERR_CUDA;
  const ff_bank_desc& d = b->d;

  G1Params prm = publish_params(b);
  prm.n_items = n;
  for (int j = 0; j < n; ++j) {
    const int a = first + j * d.anchor_stride;
    const int sl = (a / d.anchor_stride) % d.anchor_capacity;
    prm.items[j] = rot_item(frame_at(k_pre, j, b->frame_bytes), frame_at(v, j, b->frame_bytes), b->anchor_k(layer, sl),
                            b->anchor_v(layer, sl), a);
  }
  // The slots may still be read by renders or planner blocks on other streams.
  wait_stage_events(b, s, -1);
  if (b->planner_used && b->planner_stream != s) cudaStreamWaitEvent(s, b->ev_planner, 0);
  int rc = cuda_err(launch_publish(prm, 0, s), "anchor publish launch");
  if (rc != FF_OK) return rc;
  for (int j = 0; j < n; ++j) {
    const int a = first + j * d.anchor_stride;
    const int sl = (a / d.anchor_stride) % d.anchor_capacity;
    cudaEventRecord(b->ev_anchor[sl], s);
    b->anchor_stream[sl] = s;
    b->anchor_used[sl] = true;
    b->aslot(layer, sl).tag = a;
    b->aslot(layer, sl).frames = 1;
  }
  return FF_OK;
}

int ff_render_attn(ff_bank_t* b, int layer, int stage, int chunk, const void* q_pre, const void* k_pre, const void* v,
                   void* out, void* stream) {
  if (!b) return FF_ERR_ARG;
  const ff_render_call c{layer, stage, chunk, q_pre, k_pre, v, out};
  return render_calls(b, 1, &c, static_cast<cudaStream_t>(stream));
}

int ff_render_attn_batch(ff_bank_t* b, int n, const ff_render_call* calls, void* stream) {
  if (!b || !calls || n < 1 || n > kMaxBatch) return FF_ERR_ARG;
  return render_calls(b, n, calls, static_cast<cudaStream_t>(stream));
}

int ff_plan_planner_block(const ff_bank_desc* d, int block, ff_planner_plan* out) {
  if (validate_desc(d) != FF_OK || !out || block < 0 || block >= n_planner_blocks(*d)) return FF_ERR_ARG;
  plan_planner(*d, block, out);
  return FF_OK;
}

int ff_planner_attn(ff_bank_t* b, int layer, int block, const void* q_pre, const void* k_pre, const void* v,
                    void* out, void* stream) {
  if (!b || b->d.planner_history < 1 || layer < 0 || layer >= b->d.n_layers || block < 0 ||
      block >= n_planner_blocks(b->d) || !q_pre || !k_pre || !v || !out || !aligned16(q_pre) ||
      !aligned16(k_pre) || !aligned16(v) || !aligned16(out))
    return FF_ERR_ARG;
  const ff_bank_desc& d = b->d;
  ff_planner_plan pl;
  plan_planner(d, block, &pl);
  const int n_hist = pl.hist_frames;
  std::vector<int> hslots(n_hist);
  for (int j = 0; j < n_hist; ++j) {
    const int a = (pl.hist_first_block * d.planner_block + j) * d.anchor_stride;
    hslots[j] = (a / d.anchor_stride) % d.anchor_capacity;
    if (b->aslot(layer, hslots[j]).tag != a) return FF_ERR_ANCHOR_MISSING;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaSetDevice(d.device) != cudaSuccess) return FF_ERR_CUDA;
  ff_bank::Scratch& sc = b->planner;

  // RoPE of the block's Q, K, V into scratch; nothing is published
  G1Params prm = publish_params(b);
  prm.n_items = pl.n_anchors;
  for (int r = 0; r < pl.n_anchors; ++r)
    prm.items[r] = rot_item(frame_at(k_pre, r, b->frame_bytes), frame_at(v, r, b->frame_bytes),
                            sc.own_k + static_cast<size_t>(r) * b->frame_bytes,
                            sc.own_v + static_cast<size_t>(r) * b->frame_bytes, (pl.first_anchor + r) * d.anchor_stride,
                            frame_at(q_pre, r, b->frame_bytes), sc.q_rot + static_cast<size_t>(r) * b->frame_bytes);

  const long long T = static_cast<long long>(d.frame_h) * d.frame_w;
  const int nq = static_cast<int>(pl.n_anchors * T);
  AttnParams ap{};
  ap.err = b->err;
  ap.heads = d.heads;
  attn_single_group(ap, nq, 0, out);
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.head_dim)));
  KVMaps kv;
  int rc = build_segments(b, planner_segments(d, pl),
                          [&](const SegSpec& g, const void** k, const void** vv) {
                            *k = g.plane == 0 ? static_cast<const void*>(b->anchor_k(layer, g.slot)) : sc.own_k;
                            *vv = g.plane == 0 ? static_cast<const void*>(b->anchor_v(layer, g.slot)) : sc.own_v;
                          },
                          ap.groups[0], kv);
  if (rc != FF_OK) return rc;

  CUtensorMap tq;
  if ((rc = prepare_attention(b, ap, sc.q_rot, nq, sc.part_o, sc.part_ml, b->planner_part_rows, true, &tq)) != FF_OK)
    return rc;
  if (b->planner_used && b->planner_stream != s) cudaStreamWaitEvent(s, b->ev_planner, 0);
  for (int j = 0; j < n_hist; ++j)
    if (b->anchor_used[hslots[j]] && b->anchor_stream[hslots[j]] != s) cudaStreamWaitEvent(s, b->ev_anchor[hslots[j]], 0);
  if ((rc = cuda_err(launch_publish(prm, 0, s), "planner rope launch")) != FF_OK) return rc;
  if ((rc = attend(b, ap, tq, kv, s, nullptr)) != FF_OK) return rc;
  cudaEventRecord(b->ev_planner, s);
  b->planner_stream = s;
  b->planner_used = true;
  return FF_OK;
}

int ff_packed_workspace_bytes(const ff_bank_t* b, size_t* bytes) {
  if (!b || !bytes) return FF_ERR_ARG;
  const size_t frames = static_cast<size_t>(n_anchor_frames(b->d)) + b->d.total_frames;
  *bytes = (2 * frames + b->d.total_frames) * b->frame_bytes;
  return FF_OK;
}

int ff_packed_render_attn(ff_bank_t* b, const void* q_pre, const void* k_pre, const void* v, const void* anchor_k_pre,
                          const void* anchor_v, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!b || !q_pre || !k_pre || !v || !anchor_k_pre || !anchor_v || !out || !workspace || !aligned16(q_pre) ||
      !aligned16(k_pre) || !aligned16(v) || !aligned16(anchor_k_pre) || !aligned16(anchor_v) || !aligned16(out) ||
      !aligned16(workspace))
    return FF_ERR_ARG;
  const ff_bank_desc& d = b->d;
  size_t need = 0;
  ff_packed_workspace_bytes(b, &need);
  if (workspace_bytes < need) return FF_ERR_ARG;
  const int A = n_anchor_frames(d);
  const int N = d.total_frames;
  const long long T = static_cast<long long>(d.frame_h) * d.frame_w;
  if ((A + N) * T > (1ll << 30)) return FF_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaSetDevice(d.device) != cudaSuccess) return FF_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* kall = ws;                                          // [A + N frames]: anchors, then frames
  uint8_t* vall = ws + static_cast<size_t>(A + N) * b->frame_bytes;
  uint8_t* qrot = ws + 2 * static_cast<size_t>(A + N) * b->frame_bytes;  // [N frames]

  // 1. rotary encoding of every anchor and frame into the workspace (batches of kMaxItems frames)
  G1Params prm = publish_params(b);
  int rc;
  for (int f0 = 0; f0 < A + N; f0 += kMaxItems) {
    const int f1 = std::min(A + N, f0 + kMaxItems);
    int n_items = 0;
    for (int f = f0; f < f1; ++f) {
      uint8_t* dk = kall + static_cast<size_t>(f) * b->frame_bytes;
      uint8_t* dv = vall + static_cast<size_t>(f) * b->frame_bytes;
      if (f < A)
        prm.items[n_items++] = rot_item(frame_at(anchor_k_pre, f, b->frame_bytes), frame_at(anchor_v, f, b->frame_bytes),
                                        dk, dv, f * d.anchor_stride);
      else
        prm.items[n_items++] = rot_item(frame_at(k_pre, f - A, b->frame_bytes), frame_at(v, f - A, b->frame_bytes), dk,
                                        dv, f - A, frame_at(q_pre, f - A, b->frame_bytes),
                                        qrot + static_cast<size_t>(f - A) * b->frame_bytes);
    }
    prm.n_items = n_items;
    if ((rc = cuda_err(launch_publish(prm, 0, s), "packed rope launch")) != FF_OK) return rc;
  }

  // 2. block-causal attention: one query group per chunk, up to three key segments
  const int nc = n_chunks(d);
  for (int c0 = 0; c0 < nc; c0 += kMaxGroups) {
    const int c1 = std::min(nc, c0 + kMaxGroups);
    AttnParams ap{};
    ap.err = b->err;
    ap.heads = d.heads;
    ap.n_split = 1;
    ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d.head_dim)));
    ap.n_groups = c1 - c0;
    int qb = 0;
    for (int i = c0; i < c1; ++i) {
      ff_chunk_plan pl;
      plan(d, i, &pl);
      AttnGroup& g = ap.groups[i - c0];
      g.q_row0 = static_cast<int>(pl.first_frame * T);
      g.nq = static_cast<int>(pl.n_frames * T);
      g.qb0 = qb;
      g.out = out;
      g.out_row0 = g.q_row0;
      qb += (g.nq + kQBlock - 1) / kQBlock;
      g.n_seg = 0;
      int tiles = 0;
      auto add = [&](long long row0, long long rows) {
        g.seg_map[g.n_seg] = 0;
        g.seg_row0[g.n_seg] = static_cast<int>(row0);
        g.seg_rows[g.n_seg] = static_cast<int>(rows);
        g.seg_tile0[g.n_seg] = tiles;
        tiles += static_cast<int>((rows + kKTile - 1) / kKTile);
        ++g.n_seg;
      };
      for (int j = 0; j < pl.n_anchors; ++j) add((pl.anchors[j] / d.anchor_stride) * T, T);
      const int hist_first_frame = d.chunk_frames * pl.hist_first;
      add((A + hist_first_frame) * T, (pl.hist_frames + pl.n_frames) * T);
      g.n_kv = tiles;
    }
    ap.n_qb = qb;
    KVMaps kv;
    if ((rc = make_map(b, &kv.k[0], kall, static_cast<int>((A + N) * T))) != FF_OK ||
        (rc = make_map(b, &kv.v[0], vall, static_cast<int>((A + N) * T))) != FF_OK)
      return rc;
    fill_unused_maps(kv, 1);
    CUtensorMap tq;
    if ((rc = prepare_attention(b, ap, qrot, static_cast<int>(N * T), nullptr, nullptr, 0, false, &tq)) != FF_OK ||
        (rc = attend(b, ap, tq, kv, s, nullptr)) != FF_OK)
      return rc;
  }
  return FF_OK;
}

int ff_render_kernel_count(const ff_bank_t* b, int chunk, int* count) {
  if (!b || !count || chunk < 0 || chunk >= n_chunks(b->d)) return FF_ERR_ARG;
  ff_chunk_plan pl;
  plan(b->d, chunk, &pl);
  const long long T = static_cast<long long>(b->d.frame_h) * b->d.frame_w;
  const int n_qb = static_cast<int>((pl.n_frames * T + kQBlock - 1) / kQBlock);
  const int n_kv = tiles_of(chunk_segments(b->d, chunk, pl), T);
  const SplitPlan sp = plan_split(b->d.heads * n_qb, n_kv, b->sm_count, b->part_rows);
  *count = sp.n_split > 1 ? 3 : 2;
  return FF_OK;
}

int ff_bank_wait_probe(ff_bank_t* b, int limit_ms, void* stream) {
  if (!b || limit_ms < 1 || limit_ms > 10000) return FF_ERR_ARG;
  if (cudaSetDevice(b->d.device) != cudaSuccess) return FF_ERR_CUDA;
  return cuda_err(launch_wait_probe(b->err, static_cast<unsigned long long>(limit_ms) * 1000000ull,
                                    static_cast<cudaStream_t>(stream)),
                  "wait probe launch");
}

int ff_bank_set_timing(ff_bank_t* b, int enable) {
  if (!b) return FF_ERR_ARG;
  cudaSetDevice(b->d.device);
  cudaDeviceSynchronize();
  b->n_timed = 0;
  b->timing = enable != 0;
  if (b->timing && b->timed.empty()) return grow_timed(b, kTimedPool);
  return FF_OK;
}

int ff_bank_read_timing(ff_bank_t* b, ff_kernel_times* out) {
  if (!b || !out) return FF_ERR_ARG;
  std::memset(out, 0, sizeof(*out));
  for (size_t j = 0; j < b->n_timed; ++j) {
    const TimedCall& tc = b->timed[j];
    if (cudaEventSynchronize(tc.ev[3]) != cudaSuccess) return FF_ERR_CUDA;
    float a = 0, c = 0, e = 0;
    cudaEventElapsedTime(&a, tc.ev[0], tc.ev[1]);
    cudaEventElapsedTime(&c, tc.ev[1], tc.ev[2]);
    cudaEventElapsedTime(&e, tc.ev[2], tc.ev[3]);
    out->publish_ms += a;
    out->attn_ms += c;
    out->combine_ms += tc.combine ? e : 0.0;
    out->calls += tc.calls;
    out->launches += tc.launches;
  }
  return FF_OK;
}

}  // extern "C"
