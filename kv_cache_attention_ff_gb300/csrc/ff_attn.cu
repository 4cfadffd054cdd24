// Renderer bank attention on tcgen05 tensor cores.
//
// O = softmax(Q K^T / sqrt(d)) V per head over the context
// [Gamma(i) anchors; last H stage-matched chunks; own chunk] (FlashForward,
// onedev.kr/papers/332, "어떻게 동작하나", Eq. (2); no mask inside the key set).
// The context is gathered by the K/V loads themselves: its frames are read in
// place as up to kMaxSegs key segments (anchor-slot runs, stage-ring runs),
// each through its own tensor map.
// bf16 operands, fp32 accumulation in tensor memory, fp32 online softmax.
//
// One CTA per SM, 10 warps:
//   warps 0-3  softmax warpgroup 0: rows 0..127 of the current 256-row query block
//   warps 4-7  softmax warpgroup 1: rows 128..255
//   warp  8    TMA producer: Q tiles and a ring of K/V tiles
//   warp  9    TMEM allocator and single-thread MMA issuer
// Tensor memory (512 columns): S0 | S1 | O0 | O1 (S: 128 fp32 columns, O: d).
// Per key tile j the MMA thread issues S0 = Q0 K_j^T, O0 += P0 V_{j-1},
// S1 = Q1 K_j^T, O1 += P1 V_{j-1}: the tensor pipe works on one query tile's
// products while the other warpgroup turns its scores into probabilities.
// P goes through shared memory (bf16, 128-byte swizzled, K-major); V is read
// MN-major straight from its TMA tile.  The running max is only raised when
// it grows by more than 2^8 (in exp2 units), so O is rescaled rarely; the
// final normalisation uses the same stale max, which keeps the result exact
// up to rounding.
//
// Work split: a launch carries one or more query groups (a renderer call,
// each call of a stage-wavefront batch, each chunk of a packed forward), each
// with its own key segments and output.  A (head, query block) unit covers its
// group's n_kv key tiles.  The first n_whole units run as one piece each; the
// rest are cut into n_split key ranges, so that the persistent CTAs (taking
// pieces round-robin) finish together.  Units are ordered (head, query block),
// split pieces (split, unit), so concurrently running CTAs stream the same key
// tiles (L2 reuse).  Split pieces write unnormalised partials that a small
// combine kernel merges.
#include <cuda_bf16.h>

#include "ff_internal.h"
#include "ff_ptx.cuh"

namespace ff {

template <int D>
struct AttnCfg {
  static constexpr int BM = 128;
  static constexpr int BN = 128;
  static constexpr int KB = D / 64;                 // 128-byte column blocks per row
  static constexpr int BLK = 128 * 128;             // bytes of one [128 rows x 64 bf16] swizzled block
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int NST = (D == 128) ? 3 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_KV = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_BAR = OFF_KV + NST * KV_BYTES;
  static constexpr int N_BARS = 2 + 2 * NST + 10 + 1;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // barriers, TMEM slot, abort flag; 1024 B alignment slack
  static_assert(N_BARS * 8 + 8 <= 256, "barrier area");
  static_assert(SMEM <= 232448, "shared memory");
  static constexpr int TMEM_S = 0;     // S0 at 0, S1 at 128
  static constexpr int TMEM_O = 256;   // O0 at 256, O1 at 256 + D
};

constexpr int kAttnThreads = 320;
// K/V tiles are prefetched into L2 this many tiles ahead of their loads.  The
// CTAs working on one (head, key range) stream the same tiles together, so a
// tile's first touch would otherwise stall all of them on a DRAM round trip;
// tile t is prefetched by the CTA whose query block is t mod (query blocks).
constexpr int kPrefetchTiles = 6;

// Piece -> (head, group, query block of the group, key-tile range, partial
// slot: -1 for a whole unit, else the split piece's index).
struct Piece {
  int head, g, qb, kv0, kv1, part;
};

template <class P>
__device__ __forceinline__ Piece decode_piece(const P& p, int piece) {
  Piece r;
  int unit, split, ns;
  if (piece < p.n_whole) {
    unit = piece;
    split = 0;
    ns = 1;
    r.part = -1;
  } else {
    const int q = piece - p.n_whole;
    const int rest = p.heads * p.n_qb - p.n_whole;
    split = q / rest;
    unit = p.n_whole + (q - split * rest);
    ns = p.n_split;
    r.part = q;
  }
  r.head = unit / p.n_qb;
  const int lin = unit - r.head * p.n_qb;
  int g = 0;
  while (g + 1 < p.n_groups && p.groups[g + 1].qb0 <= lin) ++g;
  r.g = g;
  r.qb = lin - p.groups[g].qb0;
  const int nkv = p.groups[g].n_kv;
  r.kv0 = static_cast<int>((static_cast<long long>(split) * nkv) / ns);
  r.kv1 = static_cast<int>((static_cast<long long>(split + 1) * nkv) / ns);
  return r;
}

// Walks the key tiles of a group in order: for each tile its map, first key
// row and the number of valid keys (<= 128; the rest of the tile belongs to
// another segment or lies past the map).  Segment fields are reloaded only
// when a segment ends.
struct TileCursor {
  int s, tw, map, row0, rows, end_tile;

  __device__ __forceinline__ void load(const AttnGroup& G) {
    map = G.seg_map[s];
    row0 = G.seg_row0[s];
    rows = G.seg_rows[s];
    end_tile = (s + 1 < G.n_seg) ? G.seg_tile0[s + 1] : G.n_kv;
  }
  __device__ __forceinline__ void start(const AttnGroup& G, int t) {
    s = 0;
    while (s + 1 < G.n_seg && G.seg_tile0[s + 1] <= t) ++s;
    tw = t - G.seg_tile0[s];
    load(G);
  }
  // tile t must follow the previous call's tile
  __device__ __forceinline__ void next(const AttnGroup& G, int t, int& row, int& valid) {
    if (t == end_tile) {
      ++s;
      tw = 0;
      load(G);
    }
    row = row0 + tw * 128;
    valid = min(128, rows - tw * 128);
    ++tw;
  }
};

template <int D, class P, class KV>
__global__ void __launch_bounds__(kAttnThreads, 1)
    bank_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ KV kv,
                     const __grid_constant__ P p) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* sKV = smem + C::OFF_KV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = bars + 2 + C::NST;
  uint64_t* s_full = bars + 2 + 2 * C::NST;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* o_done = s_full + 6;
  uint64_t* o_free = s_full + 8;
  uint64_t* fin = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::N_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(s_free + t, 128);
      mbar_init(p_full + t, 128);
      mbar_init(o_done + t, 1);
      mbar_init(o_free + t, 128);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    for (int m = 0; m < KV::kMaps; ++m) {
      tma_prefetch_desc(&kv.k[m]);
      tma_prefetch_desc(&kv.v[m]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t* err = p.err;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      uint32_t n_load = 0;
      int seg = 0;
      bool ok = true;
      for (int piece = blockIdx.x; piece < p.n_pieces && ok; piece += gridDim.x, ++seg) {
        const Piece pc = decode_piece(p, piece);
        const AttnGroup& G = p.groups[pc.g];
        const int head = pc.head, kv0 = pc.kv0, kv1 = pc.kv1;
        if (seg > 0 && !(ok = mbar_wait(q_empty, (seg - 1) & 1, abort_flag, err))) break;
        mbar_expect_tx(q_full, 2 * C::Q_BYTES);
        for (int t = 0; t < 2; ++t)
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sQ + t * C::Q_BYTES + kb * C::BLK, &tmQ, head * D + kb * 64,
                        G.q_row0 + pc.qb * 256 + t * 128, q_full);
        const int n = kv1 - kv0;
        // L2 prefetch of tile u of the piece, if this CTA's query block owns it
        const int n_qb_g = (G.nq + 255) / 256;
        TileCursor pfc;
        pfc.start(G, kv0);
        auto prefetch = [&](int u) {
          int prow, pvalid;
          pfc.next(G, kv0 + u, prow, pvalid);
          if ((kv0 + u) % n_qb_g != pc.qb) return;
          for (int kb = 0; kb < C::KB; ++kb) {
            tma_prefetch_l2_2d(&kv.k[pfc.map], head * D + kb * 64, prow);
            tma_prefetch_l2_2d(&kv.v[pfc.map], head * D + kb * 64, prow);
          }
        };
        for (int u = 0; u < kPrefetchTiles && u < n; ++u) prefetch(u);
        // consumption order: K_0, then (K_j, V_{j-1}) for j >= 1, then V_{n-1}
        TileCursor kc, vc;
        kc.start(G, kv0);
        vc.start(G, kv0);
        for (int step = 0; step <= n && ok; ++step) {
          if (step + kPrefetchTiles < n) prefetch(step + kPrefetchTiles);
          for (int which = 0; which < 2; ++which) {
            const bool is_k = (which == 0);
            const int j = is_k ? step : step - 1;
            if (is_k && step == n) continue;
            if (!is_k && step == 0) continue;
            const int stage = static_cast<int>(n_load % C::NST);
            const uint32_t use = n_load / C::NST;
            if (use > 0 && !(ok = mbar_wait(kv_empty + stage, (use - 1) & 1, abort_flag, err))) break;
            mbar_expect_tx(kv_full + stage, C::KV_BYTES);
            TileCursor& cur = is_k ? kc : vc;
            int krow, kvalid;
            cur.next(G, kv0 + j, krow, kvalid);
            const CUtensorMap* map = is_k ? &kv.k[cur.map] : &kv.v[cur.map];
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(sKV + stage * C::KV_BYTES + kb * C::BLK, map, head * D + kb * 64, krow, kv_full + stage);
            ++n_load;
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0);
      constexpr uint32_t kIdescO = idesc_bf16(128, D, 1);
      const uint32_t sQa = smem_u32(sQ), sPa = smem_u32(sP), sKVa = smem_u32(sKV);
      uint32_t n_kvc = 0, n_s[2] = {0, 0}, n_pv[2] = {0, 0};
      int seg = 0;
      bool ok = true;

      // S_t = Q_t K^T for the K tile at `ka`, once softmax t has read the previous S_t
      auto s_mma = [&](int t, uint32_t ka) -> bool {
        if (n_s[t] > 0 && !mbar_wait(s_free + t, (n_s[t] - 1) & 1, abort_flag, err)) return false;
        tc_fence_after();
        const uint32_t qa = sQa + t * C::Q_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BLK + (kk & 3) * 32;
          mma_bf16_ss(tmem + C::TMEM_S + t * 128, smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), kIdescS,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full + t);
        ++n_s[t];
        return true;
      };
      // O_t (+)= P_t V for the V tile at `va`, once P_t is stored (and, for the
      // first tile of a piece, once the previous piece's O_t has been read out)
      auto pv_mma = [&](int t, uint32_t va, bool first, int head_seg) -> bool {
        if (first && head_seg > 0 && !mbar_wait(o_free + t, (head_seg - 1) & 1, abort_flag, err)) return false;
        if (!mbar_wait(p_full + t, n_pv[t] & 1, abort_flag, err)) return false;
        tc_fence_after();
        const uint32_t pa = sPa + t * C::P_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = smem_desc(pa + (kk >> 2) * C::BLK + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(va + kk * 2048, C::BLK, 1024);
          mma_bf16_ss(tmem + C::TMEM_O + t * D, ad, bd, kIdescO, (!first || kk > 0) ? 1u : 0u);
        }
        mma_commit(o_done + t);
        ++n_pv[t];
        return true;
      };
      // K/V ring entry `li` (in load order): wait for its data, return its address
      auto kv_ready = [&](uint32_t li, uint32_t& addr) -> bool {
        const int stage = static_cast<int>(li % C::NST);
        if (!mbar_wait(kv_full + stage, (li / C::NST) & 1, abort_flag, err)) return false;
        tc_fence_after();
        addr = sKVa + stage * C::KV_BYTES;
        return true;
      };
      auto kv_release = [&](uint32_t li) { mma_commit(kv_empty + static_cast<int>(li % C::NST)); };

      // Issue order per key tile j: S0(j), PV0(j-1), S1(j), PV1(j-1).  Each S
      // is issued as soon as its softmax warpgroup has read the previous one,
      // and the two query tiles' products alternate on the tensor pipe, so the
      // two softmax warpgroups run half a tile apart.
      for (int piece = blockIdx.x; piece < p.n_pieces && ok; piece += gridDim.x, ++seg) {
        const Piece pc = decode_piece(p, piece);
        const int n = pc.kv1 - pc.kv0;
        if (!(ok = mbar_wait(q_full, seg & 1, abort_flag, err))) break;
        tc_fence_after();
        uint32_t ka = 0, va = 0;
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t ek = n_kvc;  // K_j; V_{j-1} follows it in the ring
          if (!(ok = kv_ready(ek, ka) && s_mma(0, ka))) break;
          if (j >= 1 && !(ok = kv_ready(ek + 1, va) && pv_mma(0, va, j == 1, seg))) break;
          if (!(ok = s_mma(1, ka))) break;
          kv_release(ek);
          if (j == n - 1) mma_commit(q_empty);
          if (j >= 1) {
            if (!(ok = pv_mma(1, va, j == 1, seg))) break;
            kv_release(ek + 1);
          }
          n_kvc += (j >= 1) ? 2 : 1;
        }
        if (!ok) break;
        // V_{n-1}
        if (!(ok = kv_ready(n_kvc, va) && pv_mma(0, va, n == 1, seg) && pv_mma(1, va, n == 1, seg))) break;
        kv_release(n_kvc);
        ++n_kvc;
      }
      mma_commit(fin);
      mbar_wait(fin, 0, abort_flag, err);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TMEM_S + t * 128;
    const uint32_t tO = tmem + lane_off + C::TMEM_O + t * D;
    const uint32_t p_row = smem_u32(sP + t * C::P_BYTES) + (r >> 3) * 1024 + (r & 7) * 128;
    const float sl2 = p.scale_log2;
    uint32_t n_sf = 0, n_od = 0;
    bool ok = true;
    for (int piece = blockIdx.x; piece < p.n_pieces && ok; piece += gridDim.x) {
      const Piece pc = decode_piece(p, piece);
      const AttnGroup& G = p.groups[pc.g];
      const int head = pc.head, kv0 = pc.kv0;
      const int n = pc.kv1 - pc.kv0;
      float m_run = -INFINITY, l_run = 0.f;
      TileCursor cur;
      cur.start(G, kv0);
      for (int j = 0; j < n; ++j) {
        if (!(ok = mbar_wait(s_full + t, n_sf & 1, abort_flag, err))) break;
        ++n_sf;
        tc_fence_after();
        float s[128];
        tmem_ld32(tS + 0, s);
        tmem_ld32(tS + 32, s + 32);
        tmem_ld32(tS + 64, s + 64);
        tmem_ld32(tS + 96, s + 96);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free + t);
        int krow, valid;
        cur.next(G, kv0 + j, krow, valid);
        if (valid < 128) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= valid) s[c] = -INFINITY;
        }
        // row max as a tree of 3-input maxima (8 independent chains)
        float mk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = max3f(s[k], s[8 + k], s[16 + k]);
#pragma unroll
        for (int c = 24; c < 120; c += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) mk[k] = max3f(mk[k], s[c + k], s[c + 8 + k]);
#pragma unroll
        for (int k = 0; k < 8; ++k) mk[k] = fmaxf(mk[k], s[120 + k]);
        const float mx = max3f(max3f(mk[0], mk[1], mk[2]), max3f(mk[3], mk[4], mk[5]), fmaxf(mk[6], mk[7]));
        const float m_new = mx * sl2;
        const bool need = m_new > m_run + 8.0f;
        float alpha = 1.0f;
        if (need) {
          alpha = ex2_approx(m_run - m_new);
          m_run = m_new;
        }
        uint32_t pk[64];
        const float neg_m = -m_run;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float a0, a1;
          fma2(a0, a1, s[c], s[c + 1], sl2, neg_m);
          const float p0 = ex2_approx(a0);
          const float p1 = ex2_approx(a1);
          const int k = (c >> 1) & 3;
          add2(acc[2 * k], acc[2 * k + 1], p0, p1);
          pk[c >> 1] = pack_bf16x2(p0, p1);
        }
        const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        l_run = __fmaf_rn(l_run, alpha, sum);
        if (j > 0) {
          if (!(ok = mbar_wait(o_done + t, n_od & 1, abort_flag, err))) break;
          ++n_od;
          tc_fence_after();
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
              float o[32];
              tmem_ld32(tO + cc, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(tO + cc, o);
            }
            tmem_wait_st();
          }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t addr = p_row + (c >> 3) * C::BLK + (((c & 7) ^ (r & 7)) << 4);
          st_shared_v4(addr, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full + t);
      }
      if (!ok) break;
      // epilogue: wait for the last P V product
      if (!(ok = mbar_wait(o_done + t, n_od & 1, abort_flag, err))) break;
      ++n_od;
      tc_fence_after();
      const int lrow = pc.qb * 256 + t * 128 + r;  // row within the group
      if (pc.part < 0) {
        const float inv = 1.0f / l_run;
        __nv_bfloat16* dst =
            static_cast<__nv_bfloat16*>(G.out) + (static_cast<size_t>(G.out_row0 + lrow) * p.heads + head) * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tO + cc, o);
          tmem_wait_ld();
          if (lrow < G.nq) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                 pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                 pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                 pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
          }
        }
      } else {
        const size_t prow = static_cast<size_t>(pc.part) * 256 + t * 128 + r;
        float* dst = p.part_o + prow * D;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          float o[32];
          tmem_ld32(tO + cc, o);
          tmem_wait_ld();
          float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i) d4[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
        reinterpret_cast<float2*>(p.part_ml)[prow] = make_float2(m_run, l_run);
      }
      tc_fence_before();
      mbar_arrive(o_free + t);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the key-range pieces of each (head, query block): with per-piece
// running max m_s (log2 units), sum l_s and unnormalised O_s,
//   m = max m_s,  l = sum l_s 2^(m_s - m),  O = sum O_s 2^(m_s - m) / l.
// One thread per 16 output columns of a row; it issues the loads of all pieces
// before the first use, so the merge costs one round trip to L2, and a split
// unit's 256 rows take 256 / (128 / (d / 16)) blocks: one wave of 8 blocks per
// SM for the 76 split units of a 1.3B call.
constexpr int kCombineThreads = 128;
constexpr int kCombinePer = 16;  // output columns per thread

template <int D, int NS, class P>
__global__ void __launch_bounds__(kCombineThreads, NS == 2 ? 8 : 4) attn_combine_kernel(const __grid_constant__ P p) {
  constexpr int PER = kCombinePer;
  constexpr int TPR = D / PER;                     // threads per row
  constexpr int ROWS = kCombineThreads / TPR;      // rows per block
  const int rest = p.heads * p.n_qb - p.n_whole;  // split units
  const int ru = blockIdx.x;                       // index among the split units
  const int unit = p.n_whole + ru;                 // head * n_qb + linear query block
  const int head = unit / p.n_qb;
  const int lin = unit - head * p.n_qb;
  int g = 0;
  while (g + 1 < p.n_groups && p.groups[g + 1].qb0 <= lin) ++g;
  const AttnGroup& G = p.groups[g];
  const int qb = lin - G.qb0;
  const int rloc = blockIdx.y * ROWS + threadIdx.x / TPR;  // 0..255
  const int part = threadIdx.x % TPR;
  const int lrow = qb * 256 + rloc;
  if (lrow >= G.nq) return;
  const int row = G.out_row0 + lrow;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  float2 mls[NS];
  float4 os[NS][PER / 4];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    {
      const size_t piece = static_cast<size_t>(s) * rest + ru;
      mls[s] = ml[piece * 256 + rloc];
      const float4* src = reinterpret_cast<const float4*>(p.part_o + (piece * 256 + rloc) * D + part * PER);
#pragma unroll
      for (int i = 0; i < PER / 4; ++i) os[s][i] = src[i];
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int s = 0; s < NS; ++s) m = fmaxf(m, mls[s].x);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float l = 0.f;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    {
      const float w = exp2f(mls[s].x - m);
      l = __fmaf_rn(mls[s].y, w, l);
#pragma unroll
      for (int i = 0; i < PER / 4; ++i) {
        acc[4 * i] = __fmaf_rn(os[s][i].x, w, acc[4 * i]);
        acc[4 * i + 1] = __fmaf_rn(os[s][i].y, w, acc[4 * i + 1]);
        acc[4 * i + 2] = __fmaf_rn(os[s][i].z, w, acc[4 * i + 2]);
        acc[4 * i + 3] = __fmaf_rn(os[s][i].w, w, acc[4 * i + 3]);
      }
    }
  }
  const float inv = 1.0f / l;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(G.out) + (static_cast<size_t>(row) * p.heads + head) * D + part * PER;
  uint32_t w[PER / 2];
#pragma unroll
  for (int i = 0; i < PER / 2; ++i) w[i] = pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv);
#pragma unroll
  for (int i = 0; i < PER / 8; ++i)
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

size_t attention_smem_bytes(int head_dim) {
  return head_dim == 128 ? AttnCfg<128>::SMEM : AttnCfg<64>::SMEM;
}

namespace {
template <int D, class P, class KV>
cudaError_t attn_attr() {
  return cudaFuncSetAttribute(bank_attn_kernel<D, P, KV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              AttnCfg<D>::SMEM);
}

template <int D>
cudaError_t attn_attr_all() {
  cudaError_t e = attn_attr<D, AttnParamsN<1>, KVMaps>();
  if (e == cudaSuccess) e = attn_attr<D, AttnParams, KVMaps>();
  if (e == cudaSuccess) e = attn_attr<D, AttnParamsN<kMaxBatch>, KVMapsBatch>();
  return e;
}

// A copy of `p` sized for its first NG query groups.
template <int NG>
AttnParamsN<NG> first_groups(const AttnParams& p) {
  AttnParamsN<NG> q{};
  static_cast<AttnHeader&>(q) = p;
  for (int g = 0; g < NG && g < p.n_groups; ++g) q.groups[g] = p.groups[g];
  return q;
}

template <class P, class KV>
void launch_attn_p(int head_dim, const CUtensorMap& tq, const KV& kv, const P& p, int grid, cudaStream_t s) {
  if (head_dim == 128)
    bank_attn_kernel<128><<<grid, kAttnThreads, AttnCfg<128>::SMEM, s>>>(tq, kv, p);
  else
    bank_attn_kernel<64><<<grid, kAttnThreads, AttnCfg<64>::SMEM, s>>>(tq, kv, p);
}

template <int NS, class P>
void launch_combine_ns(int head_dim, const P& p, dim3 grid, cudaStream_t s) {
  if (head_dim == 128)
    attn_combine_kernel<128, NS><<<grid, kCombineThreads, 0, s>>>(p);
  else
    attn_combine_kernel<64, NS><<<grid, kCombineThreads, 0, s>>>(p);
}

template <class P>
void launch_combine_p(int head_dim, const P& p, dim3 grid, cudaStream_t s) {
  if (p.n_split == 2)
    launch_combine_ns<2>(head_dim, p, grid, s);
  else if (p.n_split == 3)
    launch_combine_ns<3>(head_dim, p, grid, s);
  else
    launch_combine_ns<kMaxSplit>(head_dim, p, grid, s);
}
}  // namespace

cudaError_t attention_configure(int head_dim) {
  return head_dim == 128 ? attn_attr_all<128>() : attn_attr_all<64>();
}

cudaError_t launch_attention(int head_dim, const CUtensorMap& tq, const KVMaps& kv, const AttnParams& p, int grid,
                             cudaStream_t s) {
  if (p.n_groups == 1)
    launch_attn_p(head_dim, tq, kv, first_groups<1>(p), grid, s);
  else
    launch_attn_p(head_dim, tq, kv, p, grid, s);
  return cudaGetLastError();
}

cudaError_t launch_attention(int head_dim, const CUtensorMap& tq, const KVMapsBatch& kv, const AttnParams& p,
                             int grid, cudaStream_t s) {
  if (p.n_groups > kMaxBatch) return cudaErrorInvalidValue;
  launch_attn_p(head_dim, tq, kv, first_groups<kMaxBatch>(p), grid, s);
  return cudaGetLastError();
}

cudaError_t launch_combine(int head_dim, const AttnParams& p, cudaStream_t s) {
  // split units x 256 rows in blocks of 128 / (d / 16) rows
  dim3 grid(p.heads * p.n_qb - p.n_whole, 256 / (kCombineThreads / (head_dim / kCombinePer)));
  if (p.n_groups == 1)
    launch_combine_p(head_dim, first_groups<1>(p), grid, s);
  else if (p.n_groups <= kMaxBatch)
    launch_combine_p(head_dim, first_groups<kMaxBatch>(p), grid, s);
  else
    launch_combine_p(head_dim, p, grid, s);
  return cudaGetLastError();
}

}  // namespace ff
