// fa_fwd.cu -- libfa: the C ABI of include/fa_fwd.h and the host code behind it (TMA
// tensor maps, argument checks, work decomposition, launches). The kernels live in
// fa_fwd_kernel.cuh (forward) and fa_bwd.cuh (backward); philox.cuh holds the dropout
// mask and sm103_ptx.cuh the PTX wrappers.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fa_fwd.h"
#include "fa_fwd_kernel.cuh"

// Fixed scratch of fa_fwd_noalloc: the stream-K workspace for callers that cannot
// allocate device memory. Every device that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

#include "fa_bwd.cuh"

// ============================================================================= host side
namespace {

using namespace fa;

// Time limit of every device-side pipeline wait, read when a kernel is launched
// (fa_set_wait_limit_us); 2 s unless the caller changes it.
std::atomic<unsigned long long> g_wait_limit_ns{FA_WAIT_LIMIT_DEFAULT_US * 1000ull};
// Debug builds only: the partial-state length the kernel is told is cut to this many floats
// (negative: no cut), so that a test can make the range checks fire with every access still
// inside the real workspace. Release builds leave it at -1.
std::atomic<long long> g_debug_part_cap{-1};
std::atomic<long long> g_launches{0};
unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [BH, N, d] 16-bit tensor (Q, K, V loads; O stores); boxes of 64 elements (128 bytes) x
// 128 rows x 1 head, 128-byte swizzle; rows past N read as zeros and are never written (never
// the next head's rows).
int make_map(CUtensorMap* m, const void* base, int d, int N, int BH, bool bf16) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return FA_ERR_TENSOR_MAP;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_TENSOR_MAP;
}

// E4M3 tensors as bytes. [BH, N, d]: boxes of 128 bytes (one row) x 128 rows x 1 head.
int make_map_u8(CUtensorMap* m, const void* base, int d, int N, int BH) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return FA_ERR_TENSOR_MAP;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)N * d};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_TENSOR_MAP;
}

// V^T as bytes, [BH, d, ldvt] with ldvt a multiple of 16: boxes of 128 keys x d rows.
int make_map_vt(CUtensorMap* m, const void* base, int d, int ldvt, int BH) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return FA_ERR_TENSOR_MAP;
  cuuint64_t dims[3] = {(cuuint64_t)ldvt, (cuuint64_t)d, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)ldvt, (cuuint64_t)ldvt * d};
  cuuint32_t box[3] = {128, (cuuint32_t)d, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_TENSOR_MAP;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
  bool attr_set[2][2][2][2][2] = {};
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (major != 10 || minor != 3) return FA_ERR_DEVICE;
    di.sms = sms;
    di.ok = true;
  }
  *out = &di;
  return FA_OK;
}

template <int D, bool BF16, bool CAUSAL, bool DROP, bool FP8 = false>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
           const CUtensorMap& mo, const Params& p, DeviceInfo* di, int grid, cudaStream_t st) {
  using LY = Layout<D, FP8 ? 1 : 2>;
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL, DROP, FP8>;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    bool& set = di->attr_set[D == 128][BF16][CAUSAL][DROP][FP8];
    if (!set) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM_BYTES) !=
          cudaSuccess)
        return FA_ERR_CUDA;
      set = true;
    }
  }
  kern<<<grid, NUM_THREADS, LY::SMEM_BYTES, st>>>(mq, mk, mv, mo, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Stream-K workspace: partial rows of every CTA, then one counter per (item, Q tile).
struct WsPlan {
  long long n_items, n_kv, W;
  int G;
  size_t part_bytes, cnt_bytes, total;
};
WsPlan ws_plan(long long BH, int Nq, int Nk, int d, int sms) {
  WsPlan w;
  w.n_items = ((long long)Nq + 2 * BM - 1) / (2 * BM) * BH;
  w.n_kv = ((long long)Nk + BN - 1) / BN;
  w.W = w.n_items * w.n_kv;
  w.G = (int)(w.W < sms ? w.W : sms);
  auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
  // [CTA][slot 2][Q tile 2][part_cols(d)][128 rows] fp32, as the kernel indexes it
  w.part_bytes = align((size_t)w.G * 2 * 2 * BM * part_cols(d) * sizeof(float));
  w.cnt_bytes = align((size_t)w.n_items * 2 * sizeof(int));
  w.total = w.part_bytes + w.cnt_bytes;
  return w;
}

// Host-side argument checks shared by the entry points (no CUDA call).
int check_args(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
               int Nq, int Nk, int d, float scale, fa_dtype dtype, bool* noop) {
  *noop = false;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (!(scale >= 0.f) || !isfinite(scale)) return FA_ERR_SCALE;
  const long long BH = (long long)B * H;
  if (BH == 0 || Nq == 0) { *noop = true; return FA_OK; }
  if (Nk == 0) return FA_ERR_EMPTY_KEYS;
  if (BH > 0x7fffffffLL) return FA_ERR_SHAPE;
  const long long n_qblk = ((long long)Nq + 2 * BM - 1) / (2 * BM);
  if (n_qblk * BH > 0x7fffffffLL) return FA_ERR_SHAPE;
  if (!Q || !K || !V || !O || !L) return FA_ERR_NULL;
  if (((uintptr_t)Q | (uintptr_t)K | (uintptr_t)V | (uintptr_t)O) & 15) return FA_ERR_ALIGN;
  if ((uintptr_t)L & 3) return FA_ERR_ALIGN;
  return FA_OK;
}

// Dropout arguments after the host checks: the 8-bit threshold t (> 0), seed and offset.
struct DropArgs {
  uint32_t t;
  unsigned long long seed;
  unsigned int offset;
};

// The 8-bit threshold of the dropout probability: t = round(p * 256); false when p is
// negative, not finite, or so close to 1 that t would be 256 (every entry dropped).
bool dropout_threshold(float p_drop, uint32_t* t) {
  if (!(p_drop >= 0.f) || !isfinite(p_drop)) return false;
  const double tt = floor((double)p_drop * 256.0 + 0.5);
  if (tt >= 256.0) return false;
  *t = (uint32_t)tt;
  return true;
}

uint32_t dropout_bias(uint32_t t) { return (0x100u - t) * 0x00010001u; }

template <bool DROP>
int dispatch(int d, bool bf16, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
             const CUtensorMap& mv, const CUtensorMap& mo, const Params& p, DeviceInfo* di, int grid,
             cudaStream_t st) {
  const int key = (d == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
  switch (key) {
    case 0: return launch<64, false, false, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 1: return launch<64, false, true, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 2: return launch<64, true, false, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 3: return launch<64, true, true, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 4: return launch<128, false, false, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 5: return launch<128, false, true, DROP>(mq, mk, mv, mo, p, di, grid, st);
    case 6: return launch<128, true, false, DROP>(mq, mk, mv, mo, p, di, grid, st);
    default: return launch<128, true, true, DROP>(mq, mk, mv, mo, p, di, grid, st);
  }
}

int run(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Nq,
        int Nk, int d, float scale, int causal, fa_dtype dtype, void* workspace,
        size_t workspace_bytes, bool use_ws, void* stream, const DropArgs* drop = nullptr) {
  bool noop = false;
  int rc = check_args(Q, K, V, O, L, B, H, Nq, Nk, d, scale, dtype, &noop);
  if (rc != FA_OK || noop) return rc;
  const long long BH = (long long)B * H;
  if (use_ws && workspace && ((uintptr_t)workspace & 255)) return FA_ERR_ALIGN;

  DeviceInfo* di = nullptr;
  rc = device_info(&di);
  if (rc != FA_OK) return rc;

  Params p;
  p.O = O;
  p.L = L;
  p.BH = (int)BH;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qblk = (int)(((long long)Nq + 2 * BM - 1) / (2 * BM));
  p.n_items = (int)(p.n_qblk * BH);
  p.n_kv_all = (Nk + BN - 1) / BN;
  p.c = scale * 1.4426950408889634f;
  p.wait_limit_ns = wait_limit_ns();
  p.streamk = 0;
  p.ws_part = nullptr;
  p.ws_cnt = nullptr;
  p.ws_part_len = p.ws_cnt_len = 0;
  int grid = p.n_items < di->sms ? p.n_items : di->sms;
  // Full attention whose items do not fill whole waves of SMs: split the key range
  // (stream-K) when the caller provides the workspace.
  if (use_ws && !causal && p.n_items % di->sms != 0) {
    const WsPlan w = ws_plan(BH, Nq, Nk, d, di->sms);
    if (!workspace || workspace_bytes < w.total) return FA_ERR_WORKSPACE;
    p.streamk = 1;
    p.ws_part = reinterpret_cast<float*>(workspace);
    p.ws_cnt = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(workspace) + w.part_bytes);
    p.ws_part_len = (long long)(w.part_bytes / sizeof(float));
    p.ws_cnt_len = (long long)(w.cnt_bytes / sizeof(int));
    const long long cap = g_debug_part_cap.load();
    if (cap >= 0 && cap < p.ws_part_len) p.ws_part_len = cap;
    grid = w.G;
  }

  p.o_scale = 1.f;
  p.drop_bias = 0;
  p.drop_offset = 0;
  p.drop_rscale = 1.f;
  p.drop_keys = philox_keys(0);
  if (drop) {
    p.drop_bias = dropout_bias(drop->t);
    p.drop_keys = philox_keys(drop->seed);
    p.drop_offset = drop->offset;
    p.drop_rscale = (float)(256.0 / (256.0 - (double)drop->t));
  }

  const bool bf16 = dtype == FA_BF16;
  CUtensorMap mq, mk, mv, mo;
  if ((rc = make_map(&mq, Q, d, Nq, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mk, K, d, Nk, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mv, V, d, Nk, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mo, O, d, Nq, (int)BH, bf16)) != FA_OK) return rc;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return drop ? dispatch<true>(d, bf16, causal, mq, mk, mv, mo, p, di, grid, st)
              : dispatch<false>(d, bf16, causal, mq, mk, mv, mo, p, di, grid, st);
}

// One thread per (row, group of 16 keys): the keep bytes of the dropout mask, computed by
// the same device functions the attention kernel uses.
__global__ void fa_dropout_mask_kernel(uint8_t* keep, long long rows, int Nq, int Nk, int groups,
                                       uint32_t bias, const __grid_constant__ PhiloxKeys keys,
                                       uint32_t offset) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= rows * groups) return;
  const long long r = t / groups;
  const int g = (int)(t % groups);
  const uint32_t bh = (uint32_t)(r / Nq), i = (uint32_t)(r % Nq);
  const uint4 w = fa::dropout_words((uint32_t)g, i, bh, offset, keys);
  uint8_t* dst = keep + r * Nk;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t f0, f1;
    fa::keep_flags4(fa::uint4_word(w, m), bias, f0, f1);
    const uint32_t flag[4] = {(f0 >> 8) & 1u, (f0 >> 24) & 1u, (f1 >> 8) & 1u, (f1 >> 24) & 1u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 16 * g + 4 * m + e;
      if (j < Nk) dst[j] = (uint8_t)flag[e];
    }
  }
}

// ------------------------------------------------------------------------ E4M3 inputs
// V [BH, Nk, d] -> V^T [BH, d, ldvt] (bytes), keys Nk..ldvt-1 zero. One block per
// (head, 64 keys): 64 rows of d = 128 bytes are staged in shared memory, then written out
// as 16-byte runs of consecutive keys.
constexpr int VT_KEYS = 64;
constexpr int VT_STRIDE = 144;  // staged row stride: 16-byte aligned, spreads the banks
__global__ void __launch_bounds__(256) fa_fp8_transpose_v_kernel(const uint8_t* V, uint8_t* Vt,
                                                                 int Nk, int ldvt) {
  constexpr int D = 128;
  __shared__ __align__(16) uint8_t tile[VT_KEYS * VT_STRIDE];
  const int bh = blockIdx.x;
  const int k0 = blockIdx.y * VT_KEYS;
  const uint8_t* src = V + (size_t)bh * Nk * D;
  uint8_t* dst = Vt + (size_t)bh * D * ldvt;
  for (int idx = threadIdx.x; idx < VT_KEYS * (D / 16); idx += blockDim.x) {
    const int row = idx / (D / 16), c16 = idx % (D / 16);
    const int key = k0 + row;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (key < Nk) v = *reinterpret_cast<const uint4*>(src + (size_t)key * D + c16 * 16);
    *reinterpret_cast<uint4*>(tile + row * VT_STRIDE + c16 * 16) = v;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < D * (VT_KEYS / 16); idx += blockDim.x) {
    const int dcol = idx / (VT_KEYS / 16), kq = idx % (VT_KEYS / 16);
    const int key = k0 + kq * 16;
    if (key >= ldvt) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) x |= (uint32_t)tile[(kq * 16 + 4 * q + e) * VT_STRIDE + dcol] << (8 * e);
      w[q] = x;
    }
    *reinterpret_cast<uint4*>(dst + (size_t)dcol * ldvt + key) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

long long fp8_ldvt(int Nk) { return ((long long)Nk + 15) / 16 * 16; }
size_t fp8_ws_bytes(long long BH, int Nk, int d) {
  return (size_t)(BH * d * fp8_ldvt(Nk) + 255) / 256 * 256;
}

int run_fp8(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Nq,
            int Nk, int d, float scale, int causal, float q_descale, float k_descale,
            float v_descale, fa_dtype out_dtype, void* workspace, size_t workspace_bytes,
            void* stream) {
  bool noop = false;
  int rc = check_args(Q, K, V, O, L, B, H, Nq, Nk, d, scale, out_dtype, &noop);
  if (rc != FA_OK || noop) return rc;
  if (d != 128) return FA_ERR_HEAD_DIM;
  for (float x : {q_descale, k_descale, v_descale})
    if (!(x > 0.f) || !isfinite(x)) return FA_ERR_SCALE;
  const long long BH = (long long)B * H;
  if (!workspace || workspace_bytes < fp8_ws_bytes(BH, Nk, d)) return FA_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 15) return FA_ERR_ALIGN;
  const double c = (double)scale * q_descale * k_descale * 1.4426950408889634;
  if (!(c < 3.0e38)) return FA_ERR_SCALE;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != FA_OK) return rc;
  const int ldvt = (int)fp8_ldvt(Nk);

  Params p;
  p.O = O;
  p.L = L;
  p.BH = (int)BH;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qblk = (int)(((long long)Nq + 2 * BM - 1) / (2 * BM));
  p.n_items = (int)(p.n_qblk * BH);
  p.n_kv_all = (Nk + BN - 1) / BN;
  p.c = (float)c;
  p.wait_limit_ns = wait_limit_ns();
  p.streamk = 0;
  p.ws_part = nullptr;
  p.ws_cnt = nullptr;
  p.ws_part_len = p.ws_cnt_len = 0;
  p.o_scale = v_descale;
  p.drop_bias = 0;
  p.drop_offset = 0;
  p.drop_rscale = 1.f;
  p.drop_keys = philox_keys(0);
  const int grid = p.n_items < di->sms ? p.n_items : di->sms;

  CUtensorMap mq, mk, mv, mo;
  if ((rc = make_map_u8(&mq, Q, d, Nq, (int)BH)) != FA_OK) return rc;
  if ((rc = make_map_u8(&mk, K, d, Nk, (int)BH)) != FA_OK) return rc;
  if ((rc = make_map_vt(&mv, workspace, d, ldvt, (int)BH)) != FA_OK) return rc;
  if ((rc = make_map(&mo, O, d, Nq, (int)BH, out_dtype == FA_BF16)) != FA_OK) return rc;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const long long kblocks = (ldvt + VT_KEYS - 1) / VT_KEYS;
  if (kblocks > 65535) return FA_ERR_SHAPE;
  const dim3 tgrid((unsigned)BH, (unsigned)kblocks);
  fa_fp8_transpose_v_kernel<<<tgrid, 256, 0, st>>>(reinterpret_cast<const uint8_t*>(V),
                                                    reinterpret_cast<uint8_t*>(workspace), Nk, ldvt);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (cudaPeekAtLastError() != cudaSuccess) return FA_ERR_CUDA;
  const int key = (out_dtype == FA_BF16 ? 2 : 0) + (causal ? 1 : 0);
  switch (key) {
    case 0: return launch<128, false, false, false, true>(mq, mk, mv, mo, p, di, grid, st);
    case 1: return launch<128, false, true, false, true>(mq, mk, mv, mo, p, di, grid, st);
    case 2: return launch<128, true, false, false, true>(mq, mk, mv, mo, p, di, grid, st);
    default: return launch<128, true, true, false, true>(mq, mk, mv, mo, p, di, grid, st);
  }
}

// ---------------------------------------------------------------------------- backward
template <int D, bool BF16, bool CAUSAL, bool DROP>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
               const CUtensorMap& mdo, BwdParams p, DeviceInfo* di, cudaStream_t st) {
  using LY = BwdLayout<D>;
  using LQ = DqLayout<D>;
  auto kq = fa_bwd_dq_kernel<D, BF16, CAUSAL, DROP>;
  auto kkv = fa_bwd_dkv_kernel<D, BF16, CAUSAL, DROP>;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, LQ::SMEM_BYTES) != cudaSuccess ||
          cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  // query tiles first: D (needed by the second kernel) and dQ
  p.n_items = p.BH * p.n_qt;
  int grid = p.n_items < di->sms ? p.n_items : di->sms;
  kq<<<grid, BW_THREADS, LQ::SMEM_BYTES, st>>>(mq, mdo, mk, mv, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (cudaPeekAtLastError() != cudaSuccess) return FA_ERR_CUDA;
  p.n_items = p.BH * p.n_kt;
  grid = p.n_items < di->sms ? p.n_items : di->sms;
  kkv<<<grid, BW_THREADS, LY::SMEM_BYTES, st>>>(mk, mv, mq, mdo, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <bool DROP>
int dispatch_bwd(int d, bool bf16, bool causal, const CUtensorMap& mq, const CUtensorMap& mk,
                 const CUtensorMap& mv, const CUtensorMap& mdo, const BwdParams& p, DeviceInfo* di,
                 cudaStream_t st) {
  const int key = (d == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
  switch (key) {
    case 0: return launch_bwd<64, false, false, DROP>(mq, mk, mv, mdo, p, di, st);
    case 1: return launch_bwd<64, false, true, DROP>(mq, mk, mv, mdo, p, di, st);
    case 2: return launch_bwd<64, true, false, DROP>(mq, mk, mv, mdo, p, di, st);
    case 3: return launch_bwd<64, true, true, DROP>(mq, mk, mv, mdo, p, di, st);
    case 4: return launch_bwd<128, false, false, DROP>(mq, mk, mv, mdo, p, di, st);
    case 5: return launch_bwd<128, false, true, DROP>(mq, mk, mv, mdo, p, di, st);
    case 6: return launch_bwd<128, true, false, DROP>(mq, mk, mv, mdo, p, di, st);
    default: return launch_bwd<128, true, true, DROP>(mq, mk, mv, mdo, p, di, st);
  }
}

size_t bwd_ws_bytes(long long BH, int Nq) {
  return (((size_t)BH * (size_t)Nq * sizeof(float)) + 255) & ~(size_t)255;
}

// Device address of the fixed scratch, looked up once per device (with that device
// current): in host code the array's name is only a host-side stand-in.
void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa_noalloc_scratch) != cudaSuccess || !ptr) return FA_ERR_CUDA;
    g_noalloc_addr[dev] = ptr;
  }
  *out = g_noalloc_addr[dev];
  return FA_OK;
}

// ------------------------------------------------------------------------ host buffers
// fa_fwd_host: chunks of heads stream through a ring of device slots in the caller's
// workspace. One library stream carries every host-to-device copy and one every
// device-to-host copy (one queue per copy direction, so that both directions run at
// once), and one stream per slot runs the slot's attention launches; per-slot events
// chain them: inputs in -> launch -> outputs out -> slot free for the next chunk.
constexpr int HOST_SLOTS = 4;
// Heads per chunk: enough for copies of at least 8 MB per tensor where the problem has the
// heads (measured on the GB300's host link with the other direction busy: 134 GB/s for 2 MB
// copies, 169 for 4 MB, 175 for 8 MB, 183 for 16 MB). The last chunk takes a quarter of
// that, so that what follows the last copy-in (its attention and its copy-out) is short.
constexpr size_t HOST_COPY_TARGET = 8u << 20;

struct HostPipe {
  bool ok = false;
  cudaStream_t h2d, d2h, comp[HOST_SLOTS];
  cudaEvent_t start, in[HOST_SLOTS], out[HOST_SLOTS], freed[HOST_SLOTS], h2d_done, d2h_done,
      comp_done[HOST_SLOTS];
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;  // held while a call enqueues its work (the streams and events are shared)

int host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ok) {
    auto mk_stream = [](cudaStream_t* st) { return cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) == cudaSuccess; };
    auto mk_event = [](cudaEvent_t* ev) { return cudaEventCreateWithFlags(ev, cudaEventDisableTiming) == cudaSuccess; };
    bool good = mk_stream(&hp.h2d) && mk_stream(&hp.d2h) && mk_event(&hp.start) &&
                mk_event(&hp.h2d_done) && mk_event(&hp.d2h_done);
    for (int s = 0; good && s < HOST_SLOTS; ++s)
      good = mk_stream(&hp.comp[s]) && mk_event(&hp.in[s]) && mk_event(&hp.out[s]) &&
             mk_event(&hp.freed[s]) && mk_event(&hp.comp_done[s]);
    if (!good) return FA_ERR_CUDA;
    hp.ok = true;
  }
  *out = &hp;
  return FA_OK;
}

struct HostChunks {
  long long hc, hc_tail, n;    // heads per chunk (slot capacity), of the last chunk; chunks
  size_t q, kv, o, l;          // bytes per head of Q (and O), of K (and V), of O, of L
  size_t off_k, off_v, off_o, off_l, slot;  // layout of one slot
  int slots;
};
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
// Heads of the chunk that starts with `rem` heads left: full chunks, then the last full
// chunk shortened so that the final one has hc_tail heads.
long long chunk_heads(long long rem, const HostChunks& c) {
  if (rem <= c.hc_tail) return rem;
  if (rem <= c.hc + c.hc_tail) return rem - c.hc_tail;
  return c.hc;
}
HostChunks host_chunks(long long BH, int Nq, int Nk, int d) {
  HostChunks c;
  c.q = (size_t)Nq * d * 2;
  c.kv = (size_t)Nk * d * 2;
  c.o = c.q;
  c.l = (size_t)Nq * 4;
  const size_t per_head = c.q < c.kv ? c.q : c.kv;
  c.hc = (long long)((HOST_COPY_TARGET + per_head - 1) / per_head);
  if (c.hc > BH) c.hc = BH;
  c.hc_tail = c.hc / 4 > 1 ? c.hc / 4 : 1;
  c.n = 0;
  for (long long h0 = 0; h0 < BH; h0 += chunk_heads(BH - h0, c)) ++c.n;
  c.off_k = align256(c.hc * c.q);
  c.off_v = c.off_k + align256(c.hc * c.kv);
  c.off_o = c.off_v + align256(c.hc * c.kv);
  c.off_l = c.off_o + align256(c.hc * c.o);
  c.slot = c.off_l + align256(c.hc * c.l);
  c.slots = (int)(c.n < HOST_SLOTS ? c.n : HOST_SLOTS);
  return c;
}

}  // namespace

extern "C" {

size_t fa_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
  const HostChunks c = host_chunks((long long)B * H, Nq, Nk, d);
  return (size_t)c.slots * c.slot;
}

int fa_fwd_host(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype, void* workspace,
                size_t workspace_bytes, void* stream) {
  bool noop = false;
  int rc = check_args(Q, K, V, O, L, B, H, Nq, Nk, d, scale, dtype, &noop);
  if (rc != FA_OK || noop) return rc;
  const long long BH = (long long)B * H;
  const HostChunks c = host_chunks(BH, Nq, Nk, d);
  if (!workspace || workspace_bytes < (size_t)c.slots * c.slot) return FA_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 255) return FA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != FA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = nullptr;
  if ((rc = host_pipe(dev, &hp)) != FA_OK) return rc;
  cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // everything starts after the work already queued on the caller's stream
  if (!ok(cudaEventRecord(hp->start, caller)) || !ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0)))
    return FA_ERR_CUDA;
  for (int s = 0; s < c.slots; ++s)
    if (!ok(cudaStreamWaitEvent(hp->comp[s], hp->start, 0))) return FA_ERR_CUDA;
  const uint8_t* hq = static_cast<const uint8_t*>(Q);
  const uint8_t* hk = static_cast<const uint8_t*>(K);
  const uint8_t* hv = static_cast<const uint8_t*>(V);
  uint8_t* ho = static_cast<uint8_t*>(O);
  uint8_t* hl = reinterpret_cast<uint8_t*>(L);
  long long h0 = 0;
  for (long long ch = 0; ch < c.n; ++ch, h0 += chunk_heads(BH - h0, c)) {
    const int s = (int)(ch % c.slots);
    uint8_t* base = static_cast<uint8_t*>(workspace) + (size_t)s * c.slot;
    const long long nh = chunk_heads(BH - h0, c);
    // inputs: once the slot's previous chunk has left it
    if (ch >= c.slots && !ok(cudaStreamWaitEvent(hp->h2d, hp->freed[s], 0))) return FA_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(base, hq + h0 * c.q, nh * c.q, cudaMemcpyHostToDevice, hp->h2d)) ||
        !ok(cudaMemcpyAsync(base + c.off_k, hk + h0 * c.kv, nh * c.kv, cudaMemcpyHostToDevice, hp->h2d)) ||
        !ok(cudaMemcpyAsync(base + c.off_v, hv + h0 * c.kv, nh * c.kv, cudaMemcpyHostToDevice, hp->h2d)) ||
        !ok(cudaEventRecord(hp->in[s], hp->h2d)))
      return FA_ERR_CUDA;
    // the attention launch on the slot's stream
    if (!ok(cudaStreamWaitEvent(hp->comp[s], hp->in[s], 0))) return FA_ERR_CUDA;
    rc = run(base, base + c.off_k, base + c.off_v, base + c.off_o,
             reinterpret_cast<float*>(base + c.off_l), 1, (int)nh, Nq, Nk, d, scale, causal, dtype,
             nullptr, 0, false, hp->comp[s]);
    if (rc != FA_OK) return rc;
    if (!ok(cudaEventRecord(hp->out[s], hp->comp[s]))) return FA_ERR_CUDA;
    // outputs
    if (!ok(cudaStreamWaitEvent(hp->d2h, hp->out[s], 0)) ||
        !ok(cudaMemcpyAsync(ho + h0 * c.o, base + c.off_o, nh * c.o, cudaMemcpyDeviceToHost, hp->d2h)) ||
        !ok(cudaMemcpyAsync(hl + h0 * c.l, base + c.off_l, nh * c.l, cudaMemcpyDeviceToHost, hp->d2h)) ||
        !ok(cudaEventRecord(hp->freed[s], hp->d2h)))
      return FA_ERR_CUDA;
  }
  // the caller's stream waits for all of it (the device-to-host stream finishes last, and
  // waiting for the others as well leaves no library work behind the caller's back)
  if (!ok(cudaEventRecord(hp->h2d_done, hp->h2d)) || !ok(cudaEventRecord(hp->d2h_done, hp->d2h)) ||
      !ok(cudaStreamWaitEvent(caller, hp->h2d_done, 0)) || !ok(cudaStreamWaitEvent(caller, hp->d2h_done, 0)))
    return FA_ERR_CUDA;
  for (int s = 0; s < c.slots; ++s)
    if (!ok(cudaEventRecord(hp->comp_done[s], hp->comp[s])) ||
        !ok(cudaStreamWaitEvent(caller, hp->comp_done[s], 0)))
      return FA_ERR_CUDA;
  return FA_OK;
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H, int Nq,
           int Nk, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, nullptr, 0, false, stream);
}

size_t fa_fwd_workspace_bytes(int B, int H, int Nq, int Nk, int d, int causal) {
  if (causal || B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
  DeviceInfo* di = nullptr;
  if (device_info(&di) != FA_OK) return 0;
  const long long BH = (long long)B * H;
  const long long n_items = ((long long)Nq + 2 * BM - 1) / (2 * BM) * BH;
  if (n_items % di->sms == 0) return 0;
  return ws_plan(BH, Nq, Nk, d, di->sms).total;
}

int fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype, void* workspace,
              size_t workspace_bytes, void* stream) {
  return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, workspace, workspace_bytes,
             true, stream);
}

int fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                   int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  bool noop = false;
  int rc = check_args(Q, K, V, O, L, B, H, Nq, Nk, d, scale, dtype, &noop);
  if (rc != FA_OK || noop) return rc;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != FA_OK) return rc;
  const long long BH = (long long)B * H;
  const long long n_items = ((long long)Nq + 2 * BM - 1) / (2 * BM) * BH;
  if (causal || n_items % di->sms == 0)  // no split of the key range: no scratch needed
    return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, nullptr, 0, false, stream);
  const WsPlan w = ws_plan(BH, Nq, Nk, d, di->sms);
  if (w.total > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch)) != FA_OK) return rc;
  // the counters must start at zero; the array keeps the previous call's contents
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(reinterpret_cast<uint8_t*>(scratch) + w.part_bytes, 0, w.cnt_bytes, st) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, scratch,
             (size_t)FA_NOALLOC_SCRATCH_BYTES, true, stream);
}

int fa_fwd_dropout(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
                   int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype, float p_drop,
                   unsigned long long seed, unsigned int offset, void* stream) {
  uint32_t t = 0;
  if (!dropout_threshold(p_drop, &t)) return FA_ERR_DROPOUT;
  if (t == 0)  // nothing is dropped: the plain forward pass
    return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, nullptr, 0, false, stream);
  const DropArgs da{t, seed, offset};
  return run(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, dtype, nullptr, 0, false, stream, &da);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Nk, int d) {
  if (B <= 0 || H <= 0 || Nk <= 0 || d != 128) return 0;
  return fp8_ws_bytes((long long)B * H, Nk, d);
}

int fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* L, int B, int H,
               int Nq, int Nk, int d, float scale, int causal, float q_descale, float k_descale,
               float v_descale, fa_dtype out_dtype, void* workspace, size_t workspace_bytes,
               void* stream) {
  return run_fp8(Q, K, V, O, L, B, H, Nq, Nk, d, scale, causal, q_descale, k_descale, v_descale,
                 out_dtype, workspace, workspace_bytes, stream);
}

int fa_dropout_mask(unsigned char* keep, int B, int H, int Nq, int Nk, float p_drop,
                    unsigned long long seed, unsigned int offset, void* stream) {
  uint32_t t = 0;
  if (!dropout_threshold(p_drop, &t)) return FA_ERR_DROPOUT;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  const long long rows = (long long)B * H * Nq;
  if (rows == 0 || Nk == 0) return FA_OK;
  if ((long long)B * H > 0x7fffffffLL) return FA_ERR_SHAPE;
  if (!keep) return FA_ERR_NULL;
  const int groups = (Nk + 15) / 16;
  const long long threads = rows * groups;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return FA_ERR_SHAPE;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc != FA_OK) return rc;
  fa_dropout_mask_kernel<<<(unsigned)grid, block, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      keep, rows, Nq, Nk, groups, dropout_bias(t), philox_keys(seed), offset);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
  return bwd_ws_bytes((long long)B * H, Nq);
}

static int run_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* L, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, fa_dtype dtype, void* workspace,
                   size_t workspace_bytes, void* stream, const DropArgs* drop) {
  bool noop = false;
  // Q, K, V as in the forward; O stands in for the output argument of the shared checks
  int rc = check_args(Q, K, V, const_cast<void*>(O), const_cast<float*>(L), B, H, Nq, Nk, d, scale,
                      dtype, &noop);
  if (rc != FA_OK) return rc;
  if (noop) return FA_OK;
  if (!dO || !dQ || !dK || !dV) return FA_ERR_NULL;
  if (((uintptr_t)dO | (uintptr_t)dQ | (uintptr_t)dK | (uintptr_t)dV) & 15) return FA_ERR_ALIGN;
  const long long BH = (long long)B * H;
  if (!workspace || workspace_bytes < bwd_ws_bytes(BH, Nq)) return FA_ERR_WORKSPACE;
  if ((uintptr_t)workspace & 15) return FA_ERR_ALIGN;
  DeviceInfo* di = nullptr;
  if ((rc = device_info(&di)) != FA_OK) return rc;
  const bool bf16 = dtype == FA_BF16;
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = make_map(&mq, Q, d, Nq, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mk, K, d, Nk, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mv, V, d, Nk, (int)BH, bf16)) != FA_OK) return rc;
  if ((rc = make_map(&mdo, dO, d, Nq, (int)BH, bf16)) != FA_OK) return rc;
  BwdParams p;
  p.O = O;
  p.dO = dO;
  p.L = L;
  p.Dws = reinterpret_cast<float*>(workspace);
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.BH = (int)BH;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qt = (Nq + BM - 1) / BM;
  p.n_kt = (Nk + BN - 1) / BN;
  p.n_items = 0;
  p.c = scale * 1.4426950408889634f;
  p.scale = scale;
  p.wait_limit_ns = wait_limit_ns();
  p.drop_bias = 0;
  p.drop_offset = 0;
  p.drop_rscale = 1.f;
  p.drop_keys = philox_keys(0);
  if (drop) {
    p.drop_bias = dropout_bias(drop->t);
    p.drop_keys = philox_keys(drop->seed);
    p.drop_offset = drop->offset;
    p.drop_rscale = (float)(256.0 / (256.0 - (double)drop->t));
  }
  if ((long long)p.n_qt * BH > 0x7fffffffLL || (long long)p.n_kt * BH > 0x7fffffffLL) return FA_ERR_SHAPE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return drop ? dispatch_bwd<true>(d, bf16, causal, mq, mk, mv, mdo, p, di, st)
              : dispatch_bwd<false>(d, bf16, causal, mq, mk, mv, mdo, p, di, st);
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
           const float* L, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d,
           float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
           void* stream) {
  return run_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                 workspace_bytes, stream, nullptr);
}

int fa_bwd_dropout(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* L, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, fa_dtype dtype, float p_drop,
                   unsigned long long seed, unsigned int offset, void* workspace,
                   size_t workspace_bytes, void* stream) {
  uint32_t t = 0;
  if (!dropout_threshold(p_drop, &t)) return FA_ERR_DROPOUT;
  if (t == 0)  // nothing was dropped: the plain backward pass
    return run_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                   workspace_bytes, stream, nullptr);
  const DropArgs da{t, seed, offset};
  return run_bwd(Q, K, V, O, dO, L, dQ, dK, dV, B, H, Nq, Nk, d, scale, causal, dtype, workspace,
                 workspace_bytes, stream, &da);
}

int fa_debug_cap_workspace(long long part_elems) {
#ifdef FA_DEBUG
  g_debug_part_cap.store(part_elems < 0 ? -1 : part_elems);
  return 1;
#else
  (void)part_elems;
  return 0;
#endif
}

int fa_last_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return v;
}

int fa_stream_status(void* stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  // queued behind the stream's work; the wait covers this stream only
  if (cudaMemcpyFromSymbolAsync(&v, g_fa_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FA_ERR_CUDA;
  return v;
}

int fa_clear_status(void) {
  const int z = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  return cudaMemcpyToSymbol(g_fa_status, &z, sizeof(int)) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_HEAD_DIM: return "head dimension d must be 64 or 128";
    case FA_ERR_SHAPE: return "B, H, Nq or Nk out of range";
    case FA_ERR_EMPTY_KEYS: return "Nk is 0 but there are query rows (softmax of an empty row)";
    case FA_ERR_SCALE: return "scale must be finite and >= 0";
    case FA_ERR_ALIGN: return "Q, K, V, O must be 16-byte aligned and L 4-byte aligned";
    case FA_ERR_DTYPE: return "dtype must be FA_F16 or FA_BF16";
    case FA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case FA_ERR_TENSOR_MAP: return "the driver rejected a TMA tensor map";
    case FA_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case FA_ERR_TIMEOUT: return "a device-side pipeline wait exceeded its time limit";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_fwd_workspace_bytes()";
    case FA_ERR_SCRATCH_LIMIT:
      return "the problem needs more scratch than fa_fwd_noalloc's fixed array (FA_NOALLOC_SCRATCH_BYTES)";
    case FA_ERR_DROPOUT:
      return "dropout probability must be finite, >= 0 and below 1 - 2^-9";
    case FA_ERR_RANGE: return "argument outside its documented range";
    case FA_ERR_BOUNDS: return "device-side: a workspace index outside its layout (debug builds check)";
    default: return "unknown status code";
  }
}

int fa_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_SHAPE;
  DeviceInfo* di = nullptr;
  int rc = device_info(&di);
  if (rc != FA_OK) return rc;
  fa::fa_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)limit_us * 1000ull);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

long long fa_num_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int fa_set_wait_limit_us(unsigned long long limit_us) {
  if (limit_us < FA_WAIT_LIMIT_MIN_US || limit_us > FA_WAIT_LIMIT_MAX_US) return FA_ERR_RANGE;
  g_wait_limit_ns.store(limit_us * 1000ull, std::memory_order_relaxed);
  return FA_OK;
}

unsigned long long fa_get_wait_limit_us(void) { return wait_limit_ns() / 1000ull; }

}  // extern "C"
