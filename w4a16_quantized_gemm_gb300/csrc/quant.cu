// Round-to-nearest INT4 quantisation of fp16 weights (the upstream step of
// the W4A16 GEMM: "LMDeploy, in depth", section "Quantization: AWQ weights
// and KV cache" names naive round-to-nearest INT4 as the baseline method; the
// codes, zeros and scales it writes are the inputs of tm_pack_weights).
//
// For every group G of g rows along K and column n (w read as exact binary32):
//   lo = min(0, min w), hi = max(0, max w); r = hi - lo, or 15 if r == 0
//   s = fp16(r / 15), at least 2^-24;  z = clamp(rint(-lo / s), 0, 15)
//   i = 1 / s;  q = clamp(rint(w * i) + z, 0, 15)
// each step one IEEE binary32 operation, round to nearest even, so the codes
// do not depend on how the work is split (one reciprocal per group and column
// keeps the per-weight work at a multiply).
//
// HBM-bound: 2 bytes read and 1 byte written per weight.  A block owns 256
// adjacent columns of one group: lane x of warp y holds 8 columns (16-byte
// loads, 8-byte code stores; a warp moves 512 contiguous bytes per row) and
// rows y, y + W, y + 2W, ... of the group (W warps), whose minima and maxima
// the warps combine through shared memory.  For g = 64 and 128 (rtn_reg_kernel,
// 8 warps) a thread keeps its g/8 rows in registers between the two passes,
// so every weight is read from HBM once; other group sizes (rtn_kernel, 4
// warps) read the group a second time, from L2.
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

// Eight codes clamp(rint(f * inv) + z, 0, 15) as bytes.  rint by the
// round-to-nearest-even of an IEEE add: for |x| < 2^22, x + 1.5 * 2^23 is
// 1.5 * 2^23 + rint(x) exactly, the integer in the low mantissa bits; the
// zero point and the clamp stay in that biased range (all exact), and the
// byte is the low bits of the pattern (no float-to-int conversion).
__device__ __forceinline__ uint2 rtn_codes(const float (&f)[kCols], const float (&inv)[kCols],
                                           const float (&zf)[kCols]) {
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  uint32_t u[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) {
    const float t = __fadd_rn(__fadd_rn(__fmul_rn(f[c], inv[c]), kMagic), zf[c]);
    u[c] = __float_as_uint(fminf(fmaxf(t, kMagic), kMagic + 15.f));
  }
  return make_uint2(__byte_perm(__byte_perm(u[0], u[1], 0x0040u), __byte_perm(u[2], u[3], 0x0040u), 0x5410u),
                    __byte_perm(__byte_perm(u[4], u[5], 0x0040u), __byte_perm(u[6], u[7], 0x0040u), 0x5410u));
}

// Per column: s (fp16 bits), z and 1/s from the group's lo and hi (the rule above).
__device__ __forceinline__ void rtn_params(const float (&lo)[kCols], const float (&hi)[kCols], float (&inv)[kCols],
                                           float (&zf)[kCols], uint32_t (&sbits)[4], uint32_t& zlo, uint32_t& zhi) {
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
  float inv[kCols], zf[kCols];
  uint32_t sbits[4], zlo, zhi;
  rtn_params(lo, hi, inv, zf, sbits, zlo, zhi);
  uint2* qr = q + (size_t)grp * g * N8 + c8;
#pragma unroll 16
  for (int k = ty; k < g; k += kRowSlices) {
    float f[kCols];
    unpack8(w[(size_t)k * N8], f);
    qr[(size_t)k * N8] = rtn_codes(f, inv, zf);
  }
  if (ty == 0) {
    z[(size_t)grp * N8 + c8] = make_uint2(zlo, zhi);
    s[(size_t)grp * N8 + c8] = make_uint4(sbits[0], sbits[1], sbits[2], sbits[3]);
  }
}

constexpr int kRegThreads = 256;
constexpr int kRegSlices = kRegThreads / kColGroups;  // 8 row slices

template <int G>
__global__ void __launch_bounds__(kRegThreads, 2) rtn_reg_kernel(const uint4* __restrict__ W, int N,
                                                               uint2* __restrict__ q, uint2* __restrict__ z,
                                                               uint4* __restrict__ s) {
  constexpr int R = G / kRegSlices;  // rows per thread
  __shared__ float s_lo[kRegSlices][kColGroups][kCols];
  __shared__ float s_hi[kRegSlices][kColGroups][kCols];
  const int tx = threadIdx.x % kColGroups, ty = threadIdx.x / kColGroups;
  const int c8 = blockIdx.x * kColGroups + tx;
  const int N8 = N / kCols;
  const bool active = c8 < N8;
  const int grp = blockIdx.y;
  const uint4* w = W + (size_t)grp * G * N8 + c8;
  uint4 v[R];
  float lo[kCols], hi[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) lo[c] = hi[c] = 0.f;
  if (active) {
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = w[(size_t)(ty + kRegSlices * i) * N8];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float f[kCols];
      unpack8(v[i], f);
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
    for (int y = 0; y < kRegSlices; ++y) {
      lo[c] = fminf(lo[c], s_lo[y][tx][c]);
      hi[c] = fmaxf(hi[c], s_hi[y][tx][c]);
    }
  float inv[kCols], zf[kCols];
  uint32_t sbits[4], zlo, zhi;
  rtn_params(lo, hi, inv, zf, sbits, zlo, zhi);
  uint2* qr = q + (size_t)grp * G * N8 + c8;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    float f[kCols];
    unpack8(v[i], f);
    qr[(size_t)(ty + kRegSlices * i) * N8] = rtn_codes(f, inv, zf);
  }
  if (ty == 0) {
    z[(size_t)grp * N8 + c8] = make_uint2(zlo, zhi);
    s[(size_t)grp * N8 + c8] = make_uint4(sbits[0], sbits[1], sbits[2], sbits[3]);
  }
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
  if (g == 128) {
    rtn_reg_kernel<128><<<grid, kRegThreads, 0, st>>>(Wv, N, qv, zv, sv);
  } else if (g == 64) {
    rtn_reg_kernel<64><<<grid, kRegThreads, 0, st>>>(Wv, N, qv, zv, sv);
  } else {
    rtn_kernel<<<grid, kQuantThreads, 0, st>>>(Wv, N, g, qv, zv, sv);
  }
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}
