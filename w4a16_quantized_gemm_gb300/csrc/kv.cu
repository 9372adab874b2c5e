// Low-bit KV cache: online quantisation of keys/values and decode attention
// that reads the int8 / int4 cache directly.
//
// The pages ("LMDeploy, in depth", section "Quantization: AWQ weights and KV
// cache"): keys and values stored as int8 or int4, quantised online,
// asymmetrically, per head and per token; the guide's "Adaptive Head
// Alignment" and "Asynchronous KV Memory Loading Pipeline" sections decode
// attention straight from the low-bit cache.  Decode attention with a few
// query heads per KV head is a streaming reduction over the cache (a few
// multiply-adds per cached byte), so it runs on the CUDA cores: the pages'
// query rearrangement exists to feed Ampere/Hopper tensor-core fragments,
// which a GEMV-shaped product does not need.
//
// Quantiser (per (token, head) vector x of D values, B = 2^bits - 1, each step
// one IEEE binary32 operation with round-to-nearest-even):
//   lo = min(0, min x), hi = max(0, max x); r = hi - lo, or B if r == 0
//   s = fp16(r / B), at least 2^-24;  z = clamp(rint(-lo / s), 0, B)
//   i = 1 / s;  q = clamp(rint(x * i) + z, 0, B)
// Codes: one byte each (int8) or two per byte, even index in the low nibble
// (int4); s fp16 and z uint8 per (token, head).
//
// Attention, one query token per sequence, D = 128, G = Hq / Hkv query heads
// per KV head: a CTA takes one (sequence, KV head) and a slice of its tokens;
// eight lanes share a token (16 head dimensions each), a warp holds four
// tokens at a time; each lane group keeps a running (max, sum, 16-dim
// accumulator) per query head (online softmax); partial states combine in
// shared memory, then over the CTAs of a thread-block cluster through
// distributed shared memory (no global scratch), and rank 0 writes the output.
#include <math_constants.h>

#include "tm_common.cuh"

namespace w4 {

namespace {

// ------------------------------------------------------------ quantiser -----

template <int EPL, int BITS>
__global__ void __launch_bounds__(128) kv_quant_kernel(const __half* __restrict__ X, long long rows,
                                                        uint8_t* __restrict__ codes, __half* __restrict__ s,
                                                        uint8_t* __restrict__ z) {
  constexpr int D = 32 * EPL;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __half* x = X + row * D + lane * EPL;
  float v[EPL];
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(x + e));
    v[e] = f.x;
    v[e + 1] = f.y;
  }
  float lo = 0.f, hi = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    lo = fminf(lo, v[e]);
    hi = fmaxf(hi, v[e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  constexpr float kB = (float)((1 << BITS) - 1);
  float r = hi - lo;
  if (r == 0.f) r = kB;
  __half sh = __float2half_rn(__fdiv_rn(r, kB));
  const __half tiny = __ushort_as_half((unsigned short)1);  // 2^-24
  if (__half2float(sh) < __half2float(tiny)) sh = tiny;
  const float sf = __half2float(sh);
  const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), kB);
  const float inv = __fdiv_rn(1.f, sf);
  uint32_t c[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) c[e] = (uint32_t)fminf(fmaxf(rintf(__fmul_rn(v[e], inv)) + zf, 0.f), kB);
  if constexpr (BITS == 8) {
    uint8_t* out = codes + row * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) *reinterpret_cast<uint16_t*>(out + e) = (uint16_t)(c[e] | (c[e + 1] << 8));
  } else {
    uint8_t* out = codes + row * (D / 2) + lane * (EPL / 2);
#pragma unroll
    for (int e = 0; e < EPL; e += 2) out[e / 2] = (uint8_t)(c[e] | (c[e + 1] << 4));
  }
  if (lane == 0) {
    s[row] = sh;
    z[row] = (uint8_t)zf;
  }
}

// ------------------------------------------------------------ attention -----

constexpr int kAttnD = 128;
constexpr int kAttnThreads = 128;  // 4 warps x 4 lane groups = 16 tokens at a time
constexpr int kSlots = kAttnThreads / 8;
constexpr int kWarps = kAttnThreads / 32;

struct AttnParams {
  const __half* Q;        // [B][Hq][D]
  const uint8_t* kc;      // [B][L][Hkv][D * BITS / 8]
  const __half* ks;       // [B][L][Hkv]
  const uint8_t* kz;
  const uint8_t* vc;
  const __half* vs;
  const uint8_t* vz;
  const int* lengths;     // [B]
  __half* out;            // [B][Hq][D]
  int L, Hq, Hkv;
};

// The 16 codes of one lane (16 bytes for int8, 8 for int4) and their
// dequantisation (q - z) * s.
template <int BITS>
__device__ __forceinline__ uint4 load_codes(const uint8_t* row, int li) {
  if constexpr (BITS == 8) {
    return *reinterpret_cast<const uint4*>(row + 16 * li);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(row + 8 * li);
    return make_uint4(u.x, u.y, 0u, 0u);
  }
}
template <int BITS>
__device__ __forceinline__ void dequant16(const uint4 u, float zf, float sf, float (&d)[16]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if constexpr (BITS == 8) {
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] = ((float)((w[i >> 2] >> (8 * (i & 3))) & 0xFFu) - zf) * sf;
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) d[i] = ((float)((w[i >> 3] >> (4 * (i & 7))) & 0xFu) - zf) * sf;
  }
}

template <int BITS, int G>
__global__ void __launch_bounds__(kAttnThreads) kv_attn_kernel(const AttnParams P) {
  constexpr int RB = kAttnD * BITS / 8;  // code bytes per (token, head)
  // per query head: running max, sum, then the 128-dim accumulator
  __shared__ float part[kWarps][G][2 + kAttnD];
  __shared__ float cta[8][G][2 + kAttnD];  // rank 0: one state per CTA of the cluster
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lg = lane >> 3, li = lane & 7;
  const int slot = warp * 4 + lg;
  const int b = blockIdx.x / P.Hkv, kvh = blockIdx.x % P.Hkv;
  const int S = gridDim.y, rank = blockIdx.y;
  const int n = max(0, min(P.lengths[b], P.L));
  const int chunk = (n + S - 1) / S;
  const int t_begin = rank * chunk, t_end = min(n, t_begin + chunk);

  // this lane's 16 query dimensions of the G heads, pre-scaled by 1 / sqrt(D)
  const float scale = rsqrtf((float)kAttnD);
  float q[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __half* qp = P.Q + ((size_t)b * P.Hq + kvh * G + h) * kAttnD + 16 * li;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(qp + i));
      q[h][i] = f.x * scale;
      q[h][i + 1] = f.y * scale;
    }
  }
  float m[G], l[G], acc[G][16];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[h][i] = 0.f;
  }
  // Codes, scales and zeros of the next PF rounds are loaded before they are
  // used, so each lane keeps PF rounds of K and V reads in flight.  The trip
  // count is warp-uniform (the score reduction shuffles across the warp); a
  // lane group whose token is past the end computes nothing.
  constexpr int PF = 4;
  uint4 kb[PF], vb[PF];
  float kzs[PF], kss[PF], vzs[PF], vss[PF];
  auto fetch = [&](int j, int tb) {
    const int t = tb + slot;
    if (t < t_end) {
      const size_t th = ((size_t)b * P.L + t) * P.Hkv + kvh;  // (token, head) index
      kb[j] = load_codes<BITS>(P.kc + th * RB, li);
      vb[j] = load_codes<BITS>(P.vc + th * RB, li);
      kzs[j] = (float)P.kz[th];
      kss[j] = __half2float(P.ks[th]);
      vzs[j] = (float)P.vz[th];
      vss[j] = __half2float(P.vs[th]);
    }
  };
#pragma unroll
  for (int j = 0; j < PF; ++j) fetch(j, t_begin + j * kSlots);
  for (int tb0 = t_begin; tb0 < t_end; tb0 += PF * kSlots) {
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      const int tb = tb0 + j * kSlots;
      if (tb >= t_end) break;  // warp-uniform
      const bool valid = tb + slot < t_end;
      float kd[16];
      if (valid) {
        dequant16<BITS>(kb[j], kzs[j], kss[j], kd);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) kd[i] = 0.f;
      }
      float sc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaf(q[h][i], kd[i], a);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        sc[h] = a;
      }
      if (valid) {
        float vd[16];
        dequant16<BITS>(vb[j], vzs[j], vss[j], vd);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(m[h], sc[h]);
          const float alpha = expf(m[h] - mn);  // 0 on the first token (m = -inf)
          const float p = expf(sc[h] - mn);
          l[h] = fmaf(l[h], alpha, p);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[h][i] = fmaf(acc[h][i], alpha, p * vd[i]);
          m[h] = mn;
        }
      }
      fetch(j, tb + PF * kSlots);
    }
  }
  // combine the 4 lane groups of each warp (lanes li, li + 8, li + 16, li + 24
  // hold the same dimensions), then the warps through shared memory
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = fmaxf(m[h], __shfl_xor_sync(0xffffffffu, m[h], 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float w = m[h] == -CUDART_INF_F ? 0.f : expf(m[h] - mx);
    float lw = l[h] * w;
    lw += __shfl_xor_sync(0xffffffffu, lw, 8);
    lw += __shfl_xor_sync(0xffffffffu, lw, 16);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float a = acc[h][i] * w;
      a += __shfl_xor_sync(0xffffffffu, a, 8);
      a += __shfl_xor_sync(0xffffffffu, a, 16);
      acc[h][i] = a;
    }
    if (lg == 0) {
      if (li == 0) {
        part[warp][h][0] = mx;
        part[warp][h][1] = lw;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) part[warp][h][2 + 16 * li + i] = acc[h][i];
    }
  }
  __syncthreads();
  // thread -> (head, dimension): G x 128 outputs over 128 threads
  float* dst_local = &cta[0][0][0];
  const uint32_t cta_base = smem_u32(dst_local);
  if (S > 1) cluster_sync_all();  // every CTA of the cluster is running before remote stores
  for (int e = threadIdx.x; e < G * (2 + kAttnD); e += kAttnThreads) {
    const int h = e / (2 + kAttnD), k = e % (2 + kAttnD);
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int s2 = 0; s2 < kWarps; ++s2) mx = fmaxf(mx, part[s2][h][0]);
    float v = 0.f;
    if (k == 0) {
      v = mx;
    } else {
#pragma unroll
      for (int s2 = 0; s2 < kWarps; ++s2) {
        const float w = part[s2][h][0] == -CUDART_INF_F ? 0.f : expf(part[s2][h][0] - mx);
        v = fmaf(part[s2][h][k], w, v);
      }
    }
    const uint32_t off = (uint32_t)(((rank * G + h) * (2 + kAttnD) + k) * 4);
    if (S > 1) {
      st_dsmem_f32(map_shared_rank(cta_base + off, 0u), v);
    } else {
      cta[0][h][k] = v;
    }
  }
  if (S > 1) {
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (rank != 0) return;
  for (int e = threadIdx.x; e < G * kAttnD; e += kAttnThreads) {
    const int h = e / kAttnD, d = e % kAttnD;
    float mx = -CUDART_INF_F;
    for (int r = 0; r < S; ++r) mx = fmaxf(mx, cta[r][h][0]);
    float num = 0.f, den = 0.f;
    if (mx != -CUDART_INF_F) {
      for (int r = 0; r < S; ++r) {
        if (cta[r][h][0] == -CUDART_INF_F) continue;
        const float w = expf(cta[r][h][0] - mx);
        den = fmaf(cta[r][h][1], w, den);
        num = fmaf(cta[r][h][2 + d], w, num);
      }
    }
    P.out[((size_t)b * P.Hq + kvh * G + h) * kAttnD + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
  }
}

template <int BITS, int G>
tm_status attn_launch(const AttnParams& P, int B, int S, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * P.Hkv), (unsigned)S, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = (unsigned)S;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = S > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kv_attn_kernel<BITS, G>, P) == cudaSuccess ? TM_OK : TM_ERR_CUDA;
}

}  // namespace

}  // namespace w4

using namespace w4;

extern "C" tm_status tm_kv_quantize(const uint16_t* X, long long rows, int D, int bits, uint8_t* codes, uint16_t* s,
                                    uint8_t* z, void* stream) {
  if (!X || !codes || !s || !z || rows < 0) return TM_ERR_INVALID_ARG;
  if ((bits != 4 && bits != 8) || (D != 64 && D != 128 && D != 256)) return TM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(X) & 3u) return TM_ERR_ALIGNMENT;
  if (bits == 8 && (reinterpret_cast<uintptr_t>(codes) & 1u)) return TM_ERR_ALIGNMENT;
  if (rows == 0) return TM_OK;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto* Xh = reinterpret_cast<const __half*>(X);
  auto* sh = reinterpret_cast<__half*>(s);
  if (bits == 8) {
    if (D == 64) kv_quant_kernel<2, 8><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
    if (D == 128) kv_quant_kernel<4, 8><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
    if (D == 256) kv_quant_kernel<8, 8><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
  } else {
    if (D == 64) kv_quant_kernel<2, 4><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
    if (D == 128) kv_quant_kernel<4, 4><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
    if (D == 256) kv_quant_kernel<8, 4><<<grid, 128, 0, st>>>(Xh, rows, codes, sh, z);
  }
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}

extern "C" tm_status tm_kv_decode_attention(const uint16_t* Q, const uint8_t* kc, const uint16_t* ks,
                                            const uint8_t* kz, const uint8_t* vc, const uint16_t* vs,
                                            const uint8_t* vz, const int* lengths, int B, int Hq, int Hkv, int L,
                                            int D, int bits, int split, uint16_t* out, void* stream) {
  if (!Q || !kc || !ks || !kz || !vc || !vs || !vz || !lengths || !out) return TM_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || L < 0 || Hq % Hkv != 0 || D != kAttnD || (bits != 4 && bits != 8))
    return TM_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4) return TM_ERR_UNSUPPORTED;
  if (split < 0 || split > 8 || (split & (split - 1))) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(out)) & 3u) return TM_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & (bits == 8 ? 15u : 7u))
    return TM_ERR_ALIGNMENT;
  if (B == 0) return TM_OK;
  int S = split;
  if (!S) {
    // enough CTAs to cover the SMs twice, each with at least 256 tokens
    const int sms = num_sms(0);
    S = 1;
    while (S < 8 && B * Hkv * S < 2 * sms && L / (2 * S) >= 256) S *= 2;
  }
  AttnParams P;
  P.Q = reinterpret_cast<const __half*>(Q);
  P.kc = kc;
  P.ks = reinterpret_cast<const __half*>(ks);
  P.kz = kz;
  P.vc = vc;
  P.vs = reinterpret_cast<const __half*>(vs);
  P.vz = vz;
  P.lengths = lengths;
  P.out = reinterpret_cast<__half*>(out);
  P.L = L;
  P.Hq = Hq;
  P.Hkv = Hkv;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  tm_status r = TM_ERR_UNSUPPORTED;
  if (bits == 8) {
    if (G == 1) r = attn_launch<8, 1>(P, B, S, st);
    if (G == 2) r = attn_launch<8, 2>(P, B, S, st);
    if (G == 4) r = attn_launch<8, 4>(P, B, S, st);
  } else {
    if (G == 1) r = attn_launch<4, 1>(P, B, S, st);
    if (G == 2) r = attn_launch<4, 2>(P, B, S, st);
    if (G == 4) r = attn_launch<4, 4>(P, B, S, st);
  }
  if (r == TM_OK) set_launch_count(1);
  return r;
}
