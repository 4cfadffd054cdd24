// ff_attention_noalloc: the attention kernel of libff for callers that cannot
// allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not an option -- inside
// a CUDA stream capture (allocation is not a capturable operation), under a
// framework that has reserved the device memory for its own caching allocator
// and forbids foreign allocations, or in a process that must not grow its
// footprint after start-up.  Such a caller already holds the rotated queries,
// the gathered key/value context and the output buffer; what the attention
// kernel still needs is scratch for the partial results of key-range splits.
// Here that scratch is one file-scope device array of fixed size, created when
// the library's module is loaded on a device and held until the process
// exits.
//
// Set-up: the first call on a device (with that device current) loads this
// module, takes the array's device address with cudaGetSymbolAddress and sets
// the attention kernel's shared-memory attribute.  Make that first call before
// any stream capture.  Later calls only enqueue work.
//
// Work plan: the same planner as the bank path (whole waves of whole units,
// then at most kMaxSplit key ranges for the rest), limited to plans whose
// partials fit the array.  The plan without any split needs no partials, so
// every problem within the kernels' index limits runs; a large problem (many
// heads, long query runs) simply runs whole units only.
//
// Sharing: every call on a device uses the same array and leaves its contents
// there.  Split partials are fully rewritten by each call before they are read;
// the kernel's error word (the array's first bytes) is cleared on the call's
// stream.  Calls whose kernels overlap on the GPU (different streams without
// ordering) race on the array and give undefined output.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ff.h"
#include "ff_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FF_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kErrBytes = 256;  // error word area at the start of the array

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int setup(int dev, void** scratch, int* sms) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FF_ERR_CUDA;
    if (major != 10 || minor != 3) return FF_ERR_UNSUPPORTED;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q{};
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return FF_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FF_ERR_CUDA;
    }
    if (ff::attention_configure(64) != cudaSuccess || ff::attention_configure(128) != cudaSuccess) return FF_ERR_CUDA;
    g_sms[dev] = count;
    g_scratch[dev] = p;
  }
  *scratch = g_scratch[dev];
  *sms = g_sms[dev];
  return FF_OK;
}

int map2d(CUtensorMap* map, const void* base, int rows, int heads, int d) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads) * d, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? FF_OK
             : FF_ERR_CUDA;
}

}  // namespace

extern "C" int ff_attention_noalloc(const void* q, const void* k, const void* v, void* out, int nq, int nk, int heads,
                                    int head_dim, void* stream) {
  if (!q || !k || !v || !out || nq < 1 || nk < 1 || heads < 1 || (head_dim != 64 && head_dim != 128))
    return FF_ERR_ARG;
  for (const void* p : {q, k, v, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return FF_ERR_ARG;
  const int n_qb = (nq + 255) / 256;
  const long long n_kv = (static_cast<long long>(nk) + 127) / 128;
  // index limits of the kernels: key tiles and (head, query block) units are ints,
  // row offsets (row * heads * head_dim) stay below 2^31 elements per tensor
  if (n_kv > (1 << 24) || static_cast<long long>(heads) * n_qb > (1 << 24) ||
      static_cast<long long>(nq) * heads * head_dim >= (1ll << 31) ||
      static_cast<long long>(nk) * heads * head_dim >= (1ll << 31))
    return FF_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FF_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int sdev = -1;
  if (cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return FF_ERR_ARG;
  }
  if (sdev != dev) return FF_ERR_ARG;  // the stream belongs to another device than the current one
  void* scratch = nullptr;
  int sms = 0;
  const int rc = setup(dev, &scratch, &sms);
  if (rc != FF_OK) return rc;

  ff::AttnParams ap{};
  ap.heads = heads;
  ff::attn_single_group(ap, nq, nk, out);
  const size_t max_part_rows = (FF_NOALLOC_SCRATCH_BYTES - kErrBytes) / (static_cast<size_t>(head_dim) * 4 + 8);
  const ff::SplitPlan sp = ff::plan_split(heads * n_qb, ap.groups[0].n_kv, sms, max_part_rows);
  ap.n_whole = sp.n_whole;
  ap.n_split = sp.n_split;
  ap.n_pieces = sp.n_pieces;
  const size_t part_rows = sp.part_rows;  // 0 without a split
  unsigned char* base = static_cast<unsigned char*>(scratch);
  ap.err = reinterpret_cast<unsigned int*>(base);
  ap.part_o = reinterpret_cast<float*>(base + kErrBytes);
  ap.part_ml = reinterpret_cast<float*>(base + kErrBytes + part_rows * head_dim * 4);
  ap.scale_log2 = static_cast<float>(1.4426950408889634 / __builtin_sqrt(static_cast<double>(head_dim)));

  CUtensorMap tq;
  ff::KVMaps kv;
  if (map2d(&tq, q, nq, heads, head_dim) != FF_OK || map2d(&kv.k[0], k, nk, heads, head_dim) != FF_OK ||
      map2d(&kv.v[0], v, nk, heads, head_dim) != FF_OK)
    return FF_ERR_CUDA;
  for (int m = 1; m < ff::kMaxMaps; ++m) {
    kv.k[m] = kv.k[0];
    kv.v[m] = kv.v[0];
  }
  if (cudaMemsetAsync(ap.err, 0, sizeof(unsigned int), s) != cudaSuccess) return FF_ERR_CUDA;
  const int grid = ap.n_pieces < sms ? ap.n_pieces : sms;
  if (ff::launch_attention(head_dim, tq, kv, ap, grid, s) != cudaSuccess) return FF_ERR_CUDA;
  if (ap.n_split > 1 && ff::launch_combine(head_dim, ap, s) != cudaSuccess) return FF_ERR_CUDA;
  return FF_OK;
}
