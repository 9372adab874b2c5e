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
// rows y, y + 4, y + 8, ... of the group, so each thread keeps a quarter of
// the group's loads in flight; the four warps combine their minima and maxima
// through shared memory.  The group is read twice, the second time from L2
// (measured faster than keeping it in shared memory, which cost occupancy).
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
  const __half tiny = __ushort_as_half((unsigned short)1);  // 2^-24, the smallest positive fp16
  float inv[kCols], zf[kCols];
  uint32_t sbits[4] = {0, 0, 0, 0}, zlo = 0, zhi = 0;
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
  uint2* qr = q + (size_t)grp * g * N8 + c8;
#pragma unroll 16
  for (int k = ty; k < g; k += kRowSlices) {
    float f[kCols];
    unpack8(w[(size_t)k * N8], f);
    uint32_t b[2] = {0, 0};
#pragma unroll
    for (int c = 0; c < kCols; ++c) {
      const float v = fminf(fmaxf(rintf(__fmul_rn(f[c], inv[c])) + zf[c], 0.f), 15.f);
      b[c >> 2] |= (uint32_t)v << (8 * (c & 3));
    }
    qr[(size_t)k * N8] = make_uint2(b[0], b[1]);
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
  rtn_kernel<<<grid, kQuantThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(W), N, g, reinterpret_cast<uint2*>(q), reinterpret_cast<uint2*>(z),
      reinterpret_cast<uint4*>(s));
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}
