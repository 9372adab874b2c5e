// Round-to-nearest INT4 quantisation of fp16 weights (the upstream step of
// the W4A16 GEMM: "LMDeploy, in depth", section "Quantization: AWQ weights
// and KV cache" names naive round-to-nearest INT4 as the baseline method; the
// codes, zeros and scales it writes are the inputs of tm_pack_weights).
//
// For every group G of g rows along K and column n (w read as exact binary32):
//   lo = min(0, min w), hi = max(0, max w); r = hi - lo, or 15 if r == 0
//   s = fp16(r / 15), at least 2^-24;  z = clamp(rint(-lo / s), 0, 15)
//   q = clamp(rint(w / s) + z, 0, 15)
// each step one IEEE binary32 operation, round to nearest even, so the codes
// do not depend on how the work is split.  The division per weight is a
// multiply by the reciprocal, computed once per group and column, plus one
// fma correction (fp16_quotient): the same codes as a division, ties included.
//
// HBM-bound: 2 bytes read and 1 byte written per weight.
// g = 64 and 128 (rtn_tma_kernel): a persistent grid, two CTAs per SM, walks
// tiles of one group's g rows x 128 columns.  One thread streams the tiles
// with 2-D TMA copies into a ring of shared-memory slots; eight warps share
// each tile, warp w rows w g/8 .. (w + 1) g/8 - 1, lane l columns 4l .. 4l+3,
// loading their rows into registers and releasing the slot at once; the
// warps' column minima and maxima meet in shared memory, each column's
// scale and zero are computed once, and each thread writes its codes as
// 4-byte stores (a warp writes 128 contiguous bytes per row).  Every weight
// is read from HBM once and the ring keeps copies in flight while the warps
// compute.  Other group sizes (rtn_kernel, 4 warps, 256 columns per block)
// read the group a second time, from L2.
#include <algorithm>

#include "tm_common.cuh"

namespace w4 {

namespace {

constexpr int kQuantThreads = 128;
constexpr int kCols = 8;        // columns per thread
constexpr int kColGroups = 32;  // 8-column groups per block (one warp wide)
constexpr int kRowSlices = kQuantThreads / kColGroups;

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[kCols]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

// Eight codes clamp(rint(f / s) + z, 0, 15) as bytes.  rint by the
// round-to-nearest-even of an IEEE add: for |x| < 2^22, x + 1.5 * 2^23 is
// 1.5 * 2^23 + rint(x) exactly, the integer in the low mantissa bits; the
// zero point and the clamp stay in that biased range (all exact), and the
// byte is the low bits of the pattern (no float-to-int conversion).
__device__ __forceinline__ uint2 rtn_codes(const float (&f)[kCols], const float (&sf)[kCols],
                                           const float (&inv)[kCols], const float (&zf)[kCols]) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  uint32_t u[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) {
    const float t = __fadd_rn(__fadd_rn(fp16_quotient(f[c], sf[c], inv[c]), kMagic), zf[c]);
    u[c] = __float_as_uint(fminf(fmaxf(t, kMagic), kMagic + 15.f));
  }
  return make_uint2(__byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u),
                    __byte_perm(__byte_perm(u[4], u[5], 0x0040u), __byte_perm(u[6], u[7], 0x0040u), 0x5410u));
}

// Per column: s (fp16 bits and value), z and 1/s from the group's lo and hi (the rule above).
__device__ __forceinline__ void rtn_params(const float (&lo)[kCols], const float (&hi)[kCols], float (&sfv)[kCols],
                                           float (&inv)[kCols], float (&zf)[kCols], uint32_t (&sbits)[4],
                                           uint32_t& zlo, uint32_t& zhi) {
  const __half tiny = __ushort_as_half((unsigned short)1);  // 2^-24, the smallest positive fp16
#pragma unroll
  for (int c = 0; c < 4; ++c) sbits[c] = 0;
  zlo = zhi = 0;
#pragma unroll
  for (int c = 0; c < kCols; ++c) {
    float r = hi[c] - lo[c];
    if (r == 0.f) r = 15.f;
    __half sh = __float2half_rn(__fdiv_rn(r, 15.f));
    if (__half2float(sh) < __half2float(tiny)) sh = tiny;
    const float sf = __half2float(sh);
    zf[c] = fminf(fmaxf(rintf(__fdiv_rn(-lo[c], sf)), 0.f), 15.f);
    sfv[c] = sf;
    inv[c] = __fdiv_rn(1.f, sf);
    sbits[c >> 1] |= (uint32_t)__half_as_ushort(sh) << (16 * (c & 1));
    if (c < 4) zlo |= (uint32_t)zf[c] << (8 * c);
    else zhi |= (uint32_t)zf[c] << (8 * (c - 4));
  }
}

__global__ void __launch_bounds__(kQuantThreads) rtn_kernel(const uint4* __restrict__ W, int N, int g,
                                                             uint2* __restrict__ q, uint2* __restrict__ z,
                                                             uint4* __restrict__ s) {
  __shared__ float s_lo[kRowSlices][kColGroups][kCols];
  __shared__ float s_hi[kRowSlices][kColGroups][kCols];
  const int tx = threadIdx.x % kColGroups, ty = threadIdx.x / kColGroups;
  const int c8 = blockIdx.x * kColGroups + tx;  // group of 8 columns
  const int N8 = N / kCols;
  const bool active = c8 < N8;
  const int grp = blockIdx.y;
  const uint4* w = W + (size_t)grp * g * N8 + c8;
  float lo[kCols], hi[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) lo[c] = hi[c] = 0.f;
  if (active) {
#pragma unroll 16
    for (int k = ty; k < g; k += kRowSlices) {
      float f[kCols];
      unpack8(w[(size_t)k * N8], f);
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        lo[c] = fminf(lo[c], f[c]);
        hi[c] = fmaxf(hi[c], f[c]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kCols; ++c) {
    s_lo[ty][tx][c] = lo[c];
    s_hi[ty][tx][c] = hi[c];
  }
  __syncthreads();
  if (!active) return;
#pragma unroll
  for (int c = 0; c < kCols; ++c)
#pragma unroll
    for (int y = 0; y < kRowSlices; ++y) {
      lo[c] = fminf(lo[c], s_lo[y][tx][c]);
      hi[c] = fmaxf(hi[c], s_hi[y][tx][c]);
    }
  float sfv[kCols], inv[kCols], zf[kCols];
  uint32_t sbits[4], zlo, zhi;
  rtn_params(lo, hi, sfv, inv, zf, sbits, zlo, zhi);
  uint2* qr = q + (size_t)grp * g * N8 + c8;
#pragma unroll 16
  for (int k = ty; k < g; k += kRowSlices) {
    float f[kCols];
    unpack8(w[(size_t)k * N8], f);
    qr[(size_t)k * N8] = rtn_codes(f, sfv, inv, zf);
  }
  if (ty == 0) {
    z[(size_t)grp * N8 + c8] = make_uint2(zlo, zhi);
    s[(size_t)grp * N8 + c8] = make_uint4(sbits[0], sbits[1], sbits[2], sbits[3]);
  }
}

static __device__ uint32_t s_err_rtn;

constexpr int kTmaCols = 128;                      // columns per tile
constexpr int kTmaWarps = 8;                       // quantising warps
constexpr int kTmaThreads = 32 * (kTmaWarps + 1);  // + one producer warp
constexpr int kTmaStages = 3;                      // ring slots

template <int G>
struct RtnTmaShape {
  static constexpr int ROWS = G / kTmaWarps;                  // rows per warp
  static constexpr uint32_t TILE = G * kTmaCols * 2;          // fp16 tile bytes
  static constexpr uint32_t RED_OFF = kTmaStages * TILE;      // [2 parity][2 lo/hi][warps][128] fp16
  static constexpr uint32_t RED = 2 * 2 * kTmaWarps * kTmaCols * 2;
  static constexpr uint32_t PAR_OFF = RED_OFF + RED;          // [2 parity][inv, zero, s][128] fp32
  static constexpr uint32_t PAR = 2 * 3 * kTmaCols * 4;
  static constexpr uint32_t BAR_OFF = PAR_OFF + PAR;          // full[S], empty[S], red[2], par[2], abort
  static constexpr uint32_t SMEM = BAR_OFF + 8 * (2 * kTmaStages + 4) + 16 + 128;  // + alignment slack
};

// One column's scale, zero point and reciprocal from the group's lo and hi
// (the rule in the header comment).
__device__ __forceinline__ void rtn_params1(float lo, float hi, float& sfv, float& inv, float& zf, __half& sh) {
  const __half tiny = __ushort_as_half((unsigned short)1);  // 2^-24, the smallest positive fp16
  float r = hi - lo;
  if (r == 0.f) r = 15.f;
  sh = __float2half_rn(__fdiv_rn(r, 15.f));
  if (__half2float(sh) < __half2float(tiny)) sh = tiny;
  const float sf = __half2float(sh);
  zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), 15.f);
  sfv = sf;
  inv = __fdiv_rn(1.f, sf);
}

// Four codes (the magic-constant rounding of rtn_codes) as the bytes of a word.
__device__ __forceinline__ uint32_t rtn_codes4(const float (&f)[4], const float (&sf)[4], const float (&inv)[4],
                                               const float (&zf)[4]) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  uint32_t u[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float t = __fadd_rn(__fadd_rn(fp16_quotient(f[c], sf[c], inv[c]), kMagic), zf[c]);
    u[c] = __float_as_uint(fminf(fmaxf(t, kMagic), kMagic + 15.f));
  }
  return __byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u);
}

__device__ __forceinline__ void unpack4(const uint2 v, float (&f)[4]) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

template <int G>
__global__ void __launch_bounds__(kTmaThreads, 2) rtn_tma_kernel(const __grid_constant__ CUtensorMap tmW, int N,
                                                                 int tiles, int NB, uint8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ z, __half* __restrict__ s) {
  using SH = RtnTmaShape<G>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 127u) & ~127u;
  uint8_t* smem = smem_raw + (base - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const uint32_t bar0 = base + SH::BAR_OFF;
  auto full = [&](int i) { return bar0 + 8 * i; };
  auto empty = [&](int i) { return bar0 + 8 * (kTmaStages + i); };
  auto red_bar = [&](int i) { return bar0 + 8 * (2 * kTmaStages + i); };
  auto par_bar = [&](int i) { return bar0 + 8 * (2 * kTmaStages + 2 + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SH::BAR_OFF + 8 * (2 * kTmaStages + 4));

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTmaStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), kTmaWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(red_bar(i), kTmaWarps);
      mbar_init(par_bar(i), kTmaWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    launch_dependents();  // the next grid may start; it waits for this one before reading q, z, s
  }
  __syncthreads();

  if (warp == kTmaWarps) {
    // ---------------- producer: one TMA copy per tile ----------------
    if (lane == 0) {
      prefetch_tmap(&tmW);
      grid_dependency_wait();  // W may be written by the preceding grid
      int issued = 0;
      for (int it = 0; it < my_tiles; ++it) {
        const int slot = it % kTmaStages;
        if (it >= kTmaStages &&
            !mbar_wait(empty(slot), (uint32_t)(it / kTmaStages - 1) & 1u, abort_flag, &s_err_rtn))
          break;
        const int t = (int)blockIdx.x + it * (int)gridDim.x;
        mbar_expect_tx(full(slot), SH::TILE);
        tma_load_2d(base + slot * SH::TILE, &tmW, (t % NB) * kTmaCols, (t / NB) * G, full(slot));
        ++issued;
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int i = max(0, issued - kTmaStages); i < issued; ++i) {
        const uint32_t bar = full(i % kTmaStages), parity = (uint32_t)(i / kTmaStages) & 1u;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(bar, parity))
          if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(&s_err_rtn, kErrTimeout);
            break;
          }
      }
    }
    return;
  }

  // ---------------- quantising warps ----------------
  // Per tile: rows into registers and the slot released; column minima and
  // maxima per warp (half2, exact) into shared memory; warp w then finishes
  // columns 16 w .. 16 w + 15 (one per lane: the three divisions of the rule
  // once per column) and publishes s, 1/s and z; every lane codes its 4 columns.
  // Both exchanges are double-buffered by tile parity behind mbarriers.
  constexpr int R = SH::ROWS;
  __half* red = reinterpret_cast<__half*>(smem + SH::RED_OFF);
  float* par = reinterpret_cast<float*>(smem + SH::PAR_OFF);
  for (int it = 0; it < my_tiles; ++it) {
    const int slot = it % kTmaStages;
    if (!mbar_wait(full(slot), (uint32_t)(it / kTmaStages) & 1u, abort_flag, &s_err_rtn)) break;
    const uint8_t* tile = smem + slot * SH::TILE;
    uint2 v[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
      v[r] = *reinterpret_cast<const uint2*>(tile + (warp * R + r) * (kTmaCols * 2) + lane * 8);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(slot));  // the rows are in registers: the slot may refill
    const __half2 zero2 = __float2half2_rn(0.f);
    __half2 lo01 = zero2, lo23 = zero2, hi01 = zero2, hi23 = zero2;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const __half2 a = *reinterpret_cast<const __half2*>(&v[r].x), b = *reinterpret_cast<const __half2*>(&v[r].y);
      lo01 = __hmin2(lo01, a);
      hi01 = __hmax2(hi01, a);
      lo23 = __hmin2(lo23, b);
      hi23 = __hmax2(hi23, b);
    }
    const int pb = it & 1;
    __half* red_lo = red + ((pb * 2 + 0) * kTmaWarps) * kTmaCols;
    __half* red_hi = red + ((pb * 2 + 1) * kTmaWarps) * kTmaCols;
    *reinterpret_cast<uint2*>(red_lo + warp * kTmaCols + 4 * lane) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo01), *reinterpret_cast<const uint32_t*>(&lo23));
    *reinterpret_cast<uint2*>(red_hi + warp * kTmaCols + 4 * lane) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&hi01), *reinterpret_cast<const uint32_t*>(&hi23));
    __syncwarp();
    if (lane == 0) mbar_arrive(red_bar(pb));
    if (!mbar_wait(red_bar(pb), (uint32_t)(it >> 1) & 1u, abort_flag, &s_err_rtn)) break;
    const int t = (int)blockIdx.x + it * (int)gridDim.x;
    const int grp = t / NB, col0 = (t % NB) * kTmaCols;
    float* p_inv = par + (pb * 3 + 0) * kTmaCols;
    float* p_zf = par + (pb * 3 + 1) * kTmaCols;
    float* p_sf = par + (pb * 3 + 2) * kTmaCols;
    if (lane < 16) {
      const int c = 16 * warp + lane;
      __half lo = red_lo[c], hi = red_hi[c];
#pragma unroll
      for (int w = 1; w < kTmaWarps; ++w) {
        lo = __hmin(lo, red_lo[w * kTmaCols + c]);
        hi = __hmax(hi, red_hi[w * kTmaCols + c]);
      }
      float sfv, inv, zf;
      __half sh;
      rtn_params1(__half2float(lo), __half2float(hi), sfv, inv, zf, sh);
      p_inv[c] = inv;
      p_zf[c] = zf;
      p_sf[c] = sfv;
      if (col0 + c < N) {
        z[(size_t)grp * N + col0 + c] = (uint8_t)zf;
        s[(size_t)grp * N + col0 + c] = sh;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(par_bar(pb));
    if (!mbar_wait(par_bar(pb), (uint32_t)(it >> 1) & 1u, abort_flag, &s_err_rtn)) break;
    const int col = col0 + 4 * lane;
    if (col < N) {
      const float4 i4 = *reinterpret_cast<const float4*>(p_inv + 4 * lane);
      const float4 z4 = *reinterpret_cast<const float4*>(p_zf + 4 * lane);
      const float4 s4 = *reinterpret_cast<const float4*>(p_sf + 4 * lane);
      const float inv[4] = {i4.x, i4.y, i4.z, i4.w}, zf[4] = {z4.x, z4.y, z4.z, z4.w};
      const float sf[4] = {s4.x, s4.y, s4.z, s4.w};
      uint8_t* qr = q + ((size_t)grp * G + warp * R) * N + col;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float f[4];
        unpack4(v[r], f);
        *reinterpret_cast<uint32_t*>(qr + (size_t)r * N) = rtn_codes4(f, sf, inv, zf);
      }
    }
  }
}

// Host side of rtn_tma_kernel: the tensor map of W (fp16 [K][N], boxes of
// 128 columns x G rows, no swizzle) and a persistent launch of at most two
// CTAs per SM, with programmatic dependent launch.
template <int G>
tm_status rtn_tma_launch(const uint16_t* W, int K, int N, uint8_t* q, uint8_t* z, uint16_t* s, cudaStream_t st) {
  using SH = RtnTmaShape<G>;
  auto kern = rtn_tma_kernel<G>;
  static std::atomic<unsigned long long> attr_done{0};  // one bit per device
  if (!smem_attr_once(attr_done, (const void*)kern, (int)SH::SMEM)) return TM_ERR_CUDA;
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return TM_ERR_CUDA;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)K};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTmaCols, (cuuint32_t)G};
  cuuint32_t es[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(W), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TM_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return TM_ERR_CUDA;
  static int per_sm_cache[64] = {};  // resident CTAs per SM, per device (0 = not yet queried)
  int per_sm = per_sm_cache[device];
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTmaThreads, SH::SMEM) != cudaSuccess ||
        per_sm < 1)
      return TM_ERR_CUDA;
    per_sm_cache[device] = per_sm;
  }
  const int NB = (N + kTmaCols - 1) / kTmaCols;
  const long long tiles_ll = (long long)NB * (K / G);
  if (tiles_ll > (1ll << 30)) return TM_ERR_UNSUPPORTED;
  const int tiles = (int)tiles_ll;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(tiles, std::min(per_sm, 2) * num_sms(device)), 1, 1);
  cfg.blockDim = dim3(kTmaThreads, 1, 1);
  cfg.dynamicSmemBytes = SH::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm, N, tiles, NB, q, z, reinterpret_cast<__half*>(s)) == cudaSuccess
             ? TM_OK
             : TM_ERR_CUDA;
}

}  // namespace

}  // namespace w4

using namespace w4;

extern "C" tm_status tm_quantize_rtn(const uint16_t* W, int K, int N, int g, uint8_t* q, uint8_t* z, uint16_t* s,
                                     void* stream) {
  if (!W || !q || !z || !s) return TM_ERR_INVALID_ARG;
  if (K <= 0 || N <= 0 || g <= 0 || K % g != 0 || N % 16 != 0 || (long long)K * N > (1ll << 34))
    return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(q) & 7u) ||
      (reinterpret_cast<uintptr_t>(z) & 7u) || (reinterpret_cast<uintptr_t>(s) & 15u))
    return TM_ERR_ALIGNMENT;
  const dim3 grid((unsigned)((N / kCols + kColGroups - 1) / kColGroups), (unsigned)(K / g));
  if (grid.y > 65535u) return TM_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto* Wv = reinterpret_cast<const uint4*>(W);
  auto* qv = reinterpret_cast<uint2*>(q);
  auto* zv = reinterpret_cast<uint2*>(z);
  auto* sv = reinterpret_cast<uint4*>(s);
  if (g == 128 || g == 64) {
    const tm_status r = g == 128 ? rtn_tma_launch<128>(W, K, N, q, z, s, st) : rtn_tma_launch<64>(W, K, N, q, z, s, st);
    if (r != TM_OK) return r;
  } else {
    rtn_kernel<<<grid, kQuantThreads, 0, st>>>(Wv, N, g, qv, zv, sv);
    if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  }
  set_launch_count(1);
  return TM_OK;
}

namespace w4 {

cudaError_t rtn_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_rtn, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_rtn, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

}  // namespace w4
