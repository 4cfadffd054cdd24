// RoPE + publish kernel (and its anchor-publish form).
//
// FlashForward renderer forward (onedev.kr/papers/332, "어떻게 동작하나", Eq. (2)):
// the chunk's own K/V are computed by the denoising forward and published into
// the stage bank, B_k^(i+1) = Tail_H(B_k^(i) U (i, K, V)); the chunk attends over
// Gamma(i) anchors, the last H stage-matched chunks and itself.  This kernel
// does the memory side of one such call:
//   * RoPE of the chunk's Q (fp32 arithmetic, bf16 out) into a scratch buffer;
//   * RoPE of the chunk's K under the published-K contract (below) and the
//     store of (K, V) into the chunk's stage-ring slot.
// The gather of [anchors; history; own] is not a copy: the attention kernel
// reads those frames where they live.  The same kernel serves anchor publishes
// (rotate at the anchor frame and store into the anchor ring), planner blocks
// and packed forwards (rotate into scratch, publishing nothing).
//
// Published-K contract: each rotated pair is
//   a' = RNE_bf16(fl64(fl64(a c) - fl64(b s))),  b' = RNE_bf16(fl64(fl64(a s) + fl64(b c)))
// with c, s the fp64 cosine/sine.  fp64 is slow on this part, so every value is
// first evaluated in fp32 with an error bound and accepted only when the whole
// error interval rounds to one bf16 value (Ziv's rounding test: monotone
// rounding of both interval ends agrees); otherwise the exact fp64 expression
// is evaluated.  Either way the result is the contract's value.
#include <cuda_bf16.h>

#include "ff_internal.h"
#include "ff_ptx.cuh"

#ifndef FF_PUB_G
#define FF_PUB_G 2
#endif

namespace ff {

// fp64 -> bf16 with one round-to-nearest-even, from the binary64 bit fields.
__device__ __forceinline__ uint32_t f64_to_bf16_rne(double v) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(v));
  const uint32_t sign = static_cast<uint32_t>(b >> 63) << 15;
  const int ex = static_cast<int>((b >> 52) & 0x7FF);
  const unsigned long long man = b & 0xFFFFFFFFFFFFFull;
  if (ex == 0x7FF) return man ? (sign | 0x7FC0u) : (sign | 0x7F80u);
  if (ex == 0) return sign;  // fp64 zero or subnormal: rounds to a signed zero
  const int e = ex - 1023;
  const unsigned long long sig = man | (1ull << 52);  // value = sig * 2^(e - 52)
  if (e >= -126) {
    unsigned long long keep = sig >> 45;  // 8 significant bits
    const unsigned long long rem = sig & ((1ull << 45) - 1);
    const unsigned long long half = 1ull << 44;
    if (rem > half || (rem == half && (keep & 1ull))) ++keep;
    int ee = e;
    if (keep == 256ull) {
      keep = 128ull;
      ++ee;
    }
    if (ee > 127) return sign | 0x7F80u;
    return sign | (static_cast<uint32_t>(ee + 127) << 7) | static_cast<uint32_t>(keep & 0x7Full);
  }
  // bf16 subnormal range: count units of 2^-133, value / 2^-133 = sig >> (-e - 81)
  const int s = -e - 81;
  if (s >= 54) return sign;
  unsigned long long keep = sig >> s;
  const unsigned long long rem = sig & ((1ull << s) - 1);
  const unsigned long long half = 1ull << (s - 1);
  if (rem > half || (rem == half && (keep & 1ull))) ++keep;
  return sign | static_cast<uint32_t>(keep);  // keep == 128 is the smallest normal
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed fp32 pairs: (r0, r1) = (a0 * b0, a1 * b1) and (a0 * b0 + c0, a1 * b1 + c1), one rounding each.
__device__ __forceinline__ void mul2v(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  unsigned long long x, y, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(d));
}
__device__ __forceinline__ void fma2v(float& r0, float& r1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  unsigned long long x, y, z, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(z) : "f"(c0), "f"(c1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(d));
}

__device__ __forceinline__ void fma2v_rm(float& r0, float& r1, float a0, float a1, float b0, float b1, float c0,
                                         float c1) {
  unsigned long long x, y, z, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(z) : "f"(c0), "f"(c1));
  asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(d));
}
__device__ __forceinline__ void fma2v_rp(float& r0, float& r1, float a0, float a1, float b0, float b1, float c0,
                                         float c1) {
  unsigned long long x, y, z, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b0), "f"(b1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(z) : "f"(c0), "f"(c1));
  asm("fma.rp.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(x), "l"(y), "l"(z));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(d));
}

// One rotated K pair, (a', b') = (a c - b s, a s + b c) with c, s the fp64
// cosine/sine, under the published-K contract; returns a' | b' << 16 (bf16).
// Fast path in fp32: p = (a c32, a s32), r = (-b s32, b c32) + p with one
// rounding (fused).  Per component, |r - contract| <= 2^-24 (3 |a||u| +
// 2 |b||w|) + 2^-51 (|a||u| + |b||w|) <= 3.0002 * 2^-24 * m, where (u, w) is
// (c, s) or (s, c) and m = |a||u32| + |b||w32| as computed (the fp32 cos/sin,
// the product and the fused sum each cost 2^-24; the contract's own fp64
// roundings ~2^-52; m itself is within 2^-22 of the exact magnitude).  The
// interval ends r -+ err are rounded outward, err = 2^-22 m + 2^-140 rounded
// up (4 * 2^-24 * m; 2^-140 covers subnormal products; m < 2^126 rules out
// overflow and NaN).  When both ends round to the same bf16 pair that pair
// is the contract's value; otherwise the fp64 expressions decide.
__device__ __forceinline__ uint32_t rot_k_pair(uint32_t kw, float2 cs, const double* cs64) {
  const float a = bf_lo(kw), b = bf_hi(kw);
  float p0, p1, r0, r1;
  mul2v(p0, p1, a, a, cs.x, cs.y);
  fma2v(r0, r1, -b, b, cs.y, cs.x, p0, p1);
  const float aa = fabsf(a), ab = fabsf(b), ac = fabsf(cs.x), as = fabsf(cs.y);
  float m0, m1, e0, e1;
  mul2v(m0, m1, ab, ab, as, ac);
  fma2v_rp(m0, m1, aa, aa, ac, as, m0, m1);
  fma2v_rp(e0, e1, m0, m1, 0x1p-22f, 0x1p-22f, 0x1p-140f, 0x1p-140f);
  float l0, l1, h0, h1;
  fma2v_rm(l0, l1, e0, e1, -1.0f, -1.0f, r0, r1);
  fma2v_rp(h0, h1, e0, e1, 1.0f, 1.0f, r0, r1);
  const uint32_t lo = pack_bf16x2(l0, l1), hi = pack_bf16x2(h0, h1);
  if (lo == hi && m0 < 0x1p126f && m1 < 0x1p126f) return lo;  // false for NaN inputs
  const double c = __ldg(cs64), s = __ldg(cs64 + 1);
  const double ad = static_cast<double>(a), bd = static_cast<double>(b);
  const uint32_t x = f64_to_bf16_rne(__dsub_rn(__dmul_rn(ad, c), __dmul_rn(bd, s)));
  const uint32_t y = f64_to_bf16_rne(__dadd_rn(__dmul_rn(ad, s), __dmul_rn(bd, c)));
  return x | (y << 16);
}

// One rotated Q pair in fp32 (bf16 out): (qa c - qb s, qa s + qb c).
__device__ __forceinline__ uint32_t rot_q_pair(uint32_t qw, float2 cs) {
  const float qa = bf_lo(qw), qb = bf_hi(qw);
  float p0, p1, r0, r1;
  mul2v(p0, p1, qa, qa, cs.x, cs.y);
  fma2v(r0, r1, -qb, qb, cs.y, cs.x, p0, p1);
  return pack_bf16x2(r0, r1);
}


__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_u4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Index of channel pair `pair` for a token at (t, y, x) in the rotary tables
// (time rows, then row-axis rows, then column-axis rows).
__device__ __forceinline__ int rope_index(const G1Header& p, int pair, int t, int y, int x) {
  if (pair < p.pt) return t * p.pt + pair;
  pair -= p.pt;
  if (pair < p.py) return p.y_base + y * p.py + pair;
  pair -= p.py;
  return p.x_base + x * p.px + pair;
}

// n / dv for 0 <= n < 2^24, dv >= 1: an fp32 reciprocal estimate (off by at
// most 2) and an exact integer correction.
__device__ __forceinline__ int div_small(int n, int dv, float inv) {
  int q = __float2int_rz(__fmul_rn(__int2float_rn(n), inv));
  int r = n - q * dv;
  while (r < 0) {
    --q;
    r += dv;
  }
  while (r >= dv) {
    ++q;
    r -= dv;
  }
  return q;
}

constexpr int kPubThreads = 128;

// Resident blocks per SM the kernel is compiled for, by heads per thread: it
// mostly waits on its loads, so occupancy is traded against registers.
template <int G>
struct PubBounds {
  static constexpr int kMinBlocks = G == 1 ? 12 : (G == 2 ? 8 : 6);
};

// A thread rotates and stores the same 16-byte unit (8 channels, 4 pairs) of
// G consecutive heads of one token: the token's position, the rotary table
// entries and the index arithmetic are shared by the G units.  Lanes run over
// the units of a head first, so each load instruction of a warp covers whole
// 128- or 256-byte head rows.
template <int N, int G>
__global__ void __launch_bounds__(kPubThreads, PubBounds<G>::kMinBlocks)
    rope_publish_kernel(const __grid_constant__ G1ParamsN<N> p) {
  const G1Item& I = p.items[blockIdx.y];
  const int upf = static_cast<int>(p.units_per_frame);
  const int tid = blockIdx.x * kPubThreads + threadIdx.x;
  if (tid >= upf / G) return;
  const uint4* src_k = static_cast<const uint4*>(I.src_k);
  const uint4* src_v = static_cast<const uint4*>(I.src_v);
  uint4* dst_k = static_cast<uint4*>(I.dst_k);
  uint4* dst_v = static_cast<uint4*>(I.dst_v);
  const bool with_q = I.src_q != nullptr;
  const uint4* q_in = static_cast<const uint4*>(I.src_q);
  uint4* q_out = static_cast<uint4*>(I.dst_q);

  const int uph = p.units_per_head;             // a power of two
  const int groups = p.units_per_row / (uph * G);  // head groups per token
  const int o = tid & (uph - 1);
  const int rest = tid >> (__ffs(uph) - 1);
  const int tok = rest / groups;
  const int off0 = tok * p.units_per_row + (rest - tok * groups) * (G * uph) + o;
  uint4 kin[G], vin[G], qin[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    kin[j] = ld_stream(src_k + off0 + j * uph);
    vin[j] = ld_stream(src_v + off0 + j * uph);
    qin[j] = with_q ? ld_stream(q_in + off0 + j * uph) : make_uint4(0, 0, 0, 0);
  }
  const int ty = div_small(tok, p.frame_w, p.inv_frame_w);
  const int tx = tok - ty * p.frame_w;
  float2 cs[4];
  const double* cs64[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int idx = rope_index(p, o * 4 + e, I.t, ty, tx);
    cs[e] = __ldg(p.rope32 + idx);
    cs64[e] = reinterpret_cast<const double*>(p.rope64 + idx);
  }
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int off = off0 + j * uph;
    const uint32_t kw[4] = {kin[j].x, kin[j].y, kin[j].z, kin[j].w};
    const uint32_t qw[4] = {qin[j].x, qin[j].y, qin[j].z, qin[j].w};
    uint32_t ko[4], qo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      ko[e] = rot_k_pair(kw[e], cs[e], cs64[e]);
      qo[e] = rot_q_pair(qw[e], cs[e]);
    }
    st_u4(dst_k + off, make_uint4(ko[0], ko[1], ko[2], ko[3]));
    st_u4(dst_v + off, vin[j]);
    if (with_q) st_u4(q_out + off, make_uint4(qo[0], qo[1], qo[2], qo[3]));
  }
}

namespace {
template <int G, class P>
void launch_publish_g(const P& p, int upf, int n_items, cudaStream_t s) {
  dim3 grid((upf / G + kPubThreads - 1) / kPubThreads, n_items);
  rope_publish_kernel<P::kItems, G><<<grid, kPubThreads, 0, s>>>(p);
}
template <class P>
void launch_publish_p(const P& p, int upf, int heads, cudaStream_t s) {
  if (heads % FF_PUB_G == 0)
    launch_publish_g<FF_PUB_G>(p, upf, p.n_items, s);
  else if (heads % 2 == 0)
    launch_publish_g<2>(p, upf, p.n_items, s);
  else
    launch_publish_g<1>(p, upf, p.n_items, s);
}
}  // namespace

namespace {
template <int N>
void launch_publish_n(const G1Params& p, int upf, int heads, cudaStream_t s) {
  G1ParamsN<N> q{};
  static_cast<G1Header&>(q) = p;
  for (int i = 0; i < p.n_items; ++i) q.items[i] = p.items[i];
  launch_publish_p(q, upf, heads, s);
}
}  // namespace

cudaError_t launch_publish(const G1Params& p, int /*grid_hint*/, cudaStream_t s) {
  const int upf = static_cast<int>(p.units_per_frame);
  const int heads = p.units_per_row / p.units_per_head;
  if (p.n_items <= kFewItems)
    launch_publish_n<kFewItems>(p, upf, heads, s);
  else if (p.n_items <= kBatchItems)
    launch_publish_n<kBatchItems>(p, upf, heads, s);
  else
    launch_publish_p(p, upf, heads, s);
  return cudaGetLastError();
}

}  // namespace ff
