// Low-bit KV cache: online quantisation of keys/values and decode attention
// that reads the int8 / int4 cache directly.
//
// The pages ("LMDeploy, in depth", section "Quantization: AWQ weights and KV
// cache"): keys and values stored as int8 or int4, quantised online,
// asymmetrically, per head and per token; the guide's "Adaptive Head
// Alignment" and "Asynchronous KV Memory Loading Pipeline" sections compute
// attention on tensor cores straight from the low-bit cache, rearranging the
// query once so that its fragments line up with the low-bit key tiles.  Here
// the same idea on mma.m16n8k16 (see the tensor-core section below): the
// codes become exact fp16 integers with one byte-permute and one subtract per
// pair, scales and zero points are applied per token outside the products.
//
// Quantiser (per (token, head) vector x of D values, B = 2^bits - 1, each step
// one IEEE binary32 operation with round-to-nearest-even):
//   lo = min(0, min x), hi = max(0, max x); r = hi - lo, or B if r == 0
//   s = fp16(r / B), at least 2^-24;  z = clamp(rint(-lo / s), 0, B)
//   i = 1 / s;  q = clamp(rint(x * i) + z, 0, B)
// Codes: one byte each (int8) or two per byte, even index in the low nibble
// (int4); s fp16 and z uint8 per (token, head).  Keys stay token-major; values
// are re-laid dimension-major in 16-token tiles (tm_kv_pack_v) for the P V
// product.
//
// Attention, one query token per sequence, D = 128, G = Hq / Hkv query heads
// per KV head: a CTA takes one (sequence, KV head) and a slice of its tokens,
// a warp a 16-token tile at a time with an online softmax per head; the warps'
// states combine in shared memory, then over the CTAs of a thread-block
// cluster through distributed shared memory (no global scratch), and rank 0
// writes the output.
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
constexpr int kAttnThreads = 128;  // 4 warps, a 16-token tile each at a time
constexpr int kWarps = kAttnThreads / 32;
// CTAs per cluster along the tokens; the combine buffer holds one state per CTA
// and must stay within the 48 KB of static shared memory.
__host__ __device__ constexpr int max_split(int G) { return G == 8 ? 4 : 8; }

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

// Combine the per-warp softmax states in `part` (max, sum, 128-dim accumulator
// per query head) into one per CTA, then over the CTAs of the cluster through
// distributed shared memory into rank 0, which writes out = acc / sum.
template <int G>
__device__ __forceinline__ void finish_attention(float (*part)[G][2 + kAttnD], float (*cta)[G][2 + kAttnD],
                                                 const AttnParams& P, int b, int kvh, int S, int rank) {
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


// ------------------------------------------------ tensor-core attention -----
//
// Per warp a tile of 16 tokens.  Scores S^T = Q K^T on mma.m16n8k16: A = the
// query heads (G of 16 rows used), B = the key codes as exact fp16 integers
// (the fp16 pattern of 1024 OR-ed with a code, minus 1024), so
// score = s_k (Q . c - z_k sum Q) / sqrt(D) per token in fp32 afterwards.  The
// k order inside every 16-dimension slice is permuted the same way on Q and K
// (slots 2t, 2t+1, 2t+8, 2t+9 hold dimensions 4t .. 4t+3), so a lane reads
// its key bytes with one 4-byte (int8) or 2-byte (int4) load.  Within the
// tile, the first n8 block holds tokens {0,1,4,5,8,9,12,13} and the second
// {2,3,6,7,10,11,14,15}: then the score fragment of a lane (head gr, tokens
// 4t .. 4t+3) is exactly its A fragment of P for out = P V (tokens 4t .. 4t+3
// in slots 2t, 2t+1, 2t+8, 2t+9).  P carries the per-token value scale
// (rounded once to fp16); V codes come from tiles stored dimension-major
// ([128 dims][16 tokens], written by tm_kv_pack_v), one 4- or 2-byte load per
// lane and n8 block of dimensions; the value zero point is removed once per
// head at the end (sum_t P_t z_t).

// Two codes -> two exact fp16 values (int8: bytes i, i+1 of w; int4: both
// nibbles of byte i of w).
template <int BITS>
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t w, int i) {
  if constexpr (BITS == 8) {
    const uint32_t x = __byte_perm(w, 0x6464u, i == 0 ? 0x4140u : 0x4342u);  // (1024 + c0, 1024 + c1)
    return hsub2_u32(x, 0x64006400u);
  } else {
    const uint32_t x = __byte_perm(w, 0u, i == 0 ? 0x4040u : 0x4141u);       // byte i in bytes 0 and 2
    const uint32_t y = lop3<0xEA>(x, 0x00F0000Fu, 0x64006400u);              // (1024 + lo, 1024 + 16 hi)
    return hfma2_u32(y, 0x2C003C00u, 0xD400E400u);                          // (x - 1024, x / 16 - 64)
  }
}

template <int BITS, int G>
__global__ void __launch_bounds__(kAttnThreads) kv_attn_tc_kernel(const AttnParams P) {
  constexpr int RB = kAttnD * BITS / 8;  // key code bytes per (token, head)
  constexpr int TB = 16 * BITS / 8;      // value tile bytes per dimension (16 tokens)
  __shared__ float part[kWarps][G][2 + kAttnD];
  __shared__ float cta[max_split(G)][G][2 + kAttnD];  // rank 0: one state per CTA of the cluster
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  const int b = blockIdx.x / P.Hkv, kvh = blockIdx.x % P.Hkv;
  const int S = gridDim.y, rank = blockIdx.y;
  const int n = max(0, min(P.lengths[b], P.L));
  const int chunk = ((n + S - 1) / S + 15) & ~15;  // whole 16-token tiles per CTA
  const int t_begin = min(n, rank * chunk), t_end = min(n, t_begin + chunk);
  const bool head = gr < G;

  // A fragments of Q (rows gr < G), permuted k order; and sum_d Q[gr][d]
  uint32_t qa[8][2];
  float qsum = 0.f;
#pragma unroll
  for (int sl = 0; sl < 8; ++sl) {
    uint2 v = make_uint2(0u, 0u);
    if (head) v = *reinterpret_cast<const uint2*>(P.Q + ((size_t)b * P.Hq + kvh * G + gr) * kAttnD + 16 * sl + 4 * t);
    qa[sl][0] = v.x;
    qa[sl][1] = v.y;
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    qsum += (f0.x + f0.y) + (f1.x + f1.y);
  }
  qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
  qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
  const float scale = rsqrtf((float)kAttnD);

  float m = -CUDART_INF_F, lp = 0.f, zc = 0.f;  // running max; this lane's partial sums
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;

  const size_t tiles_per_seq = (size_t)P.L / 16;
  for (int t0 = t_begin + 16 * warp; t0 < t_end; t0 += 16 * kWarps) {
    // ---- scores: two n8 blocks of tokens
    float r[4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int tok = t0 + 4 * (gr >> 1) + (gr & 1) + 2 * nb;  // this lane's B row (token)
      const uint8_t* krow = P.kc + (((size_t)b * P.L + tok) * P.Hkv + kvh) * RB;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int sl = 0; sl < 8; ++sl) {
        uint32_t w;
        if constexpr (BITS == 8) {
          w = *reinterpret_cast<const uint32_t*>(krow + 16 * sl + 4 * t);
        } else {
          w = *reinterpret_cast<const uint16_t*>(krow + 8 * sl + 2 * t);
        }
        const uint32_t a[4] = {qa[sl][0], 0u, qa[sl][1], 0u};
        mma_16816(d, a, codes_to_half2<BITS>(w, 0), codes_to_half2<BITS>(w, 1));
      }
      r[2 * nb] = d[0];      // token 4t + 2 nb
      r[2 * nb + 1] = d[1];  // token 4t + 2 nb + 1
    }
    float sc[4], vsc[4], vzp[4];
    float mt = -CUDART_INF_F;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = t0 + 4 * t + i;
      if (tok < t_end) {
        const size_t th = ((size_t)b * P.L + tok) * P.Hkv + kvh;
        sc[i] = __half2float(P.ks[th]) * fmaf(-(float)P.kz[th], qsum, r[i]) * scale;
        vsc[i] = __half2float(P.vs[th]);
        vzp[i] = (float)P.vz[th];
      } else {
        sc[i] = -CUDART_INF_F;
        vsc[i] = 0.f;
        vzp[i] = 0.f;
      }
      mt = fmaxf(mt, sc[i]);
    }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float mn = fmaxf(m, mt);  // finite: every tile holds at least one valid token
    const float alpha = expf(m - mn);  // 0 on the first tile (m = -inf)
    m = mn;
    __half ph[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float p = expf(sc[i] - mn);
      lp = fmaf(lp, i == 0 ? alpha : 1.f, p);
      ph[i] = __float2half_rn(p * vsc[i]);
    }
    zc = fmaf(zc, alpha, __half2float(ph[0]) * vzp[0] + __half2float(ph[1]) * vzp[1] +
                             __half2float(ph[2]) * vzp[2] + __half2float(ph[3]) * vzp[3]);
    const uint32_t pa[4] = {(uint32_t)__half_as_ushort(ph[0]) | ((uint32_t)__half_as_ushort(ph[1]) << 16), 0u,
                            (uint32_t)__half_as_ushort(ph[2]) | ((uint32_t)__half_as_ushort(ph[3]) << 16), 0u};
    // ---- out += P V over 16 n8 blocks of dimensions
    const uint8_t* vt = P.vc + (((size_t)b * P.Hkv + kvh) * tiles_per_seq + t0 / 16) * kAttnD * TB;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= alpha;
      o[j][1] *= alpha;
      uint32_t w;
      if constexpr (BITS == 8) {
        w = *reinterpret_cast<const uint32_t*>(vt + (8 * j + gr) * TB + 4 * t);
      } else {
        w = *reinterpret_cast<const uint16_t*>(vt + (8 * j + gr) * TB + 2 * t);
      }
      mma_16816(o[j], pa, codes_to_half2<BITS>(w, 0), codes_to_half2<BITS>(w, 1));
    }
  }
  // lane (gr, t): head gr, dimensions 8 j + 2 t, 8 j + 2 t + 1
  lp += __shfl_xor_sync(0xffffffffu, lp, 1);
  lp += __shfl_xor_sync(0xffffffffu, lp, 2);
  zc += __shfl_xor_sync(0xffffffffu, zc, 1);
  zc += __shfl_xor_sync(0xffffffffu, zc, 2);
  if (head) {
    if (t == 0) {
      part[warp][gr][0] = m;
      part[warp][gr][1] = lp;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      part[warp][gr][2 + 8 * j + 2 * t] = o[j][0] - zc;
      part[warp][gr][2 + 8 * j + 2 * t + 1] = o[j][1] - zc;
    }
  }
  finish_attention<G>(part, cta, P, b, kvh, S, rank);
}

// Value codes token-major [B][L][Hkv][D bytes] -> dimension-major tiles
// [B][Hkv][L/16][D][16 tokens] (int8) or [..][D][8 bytes] (int4, tokens
// 2k and 2k+1 in the low and high nibble of byte k).
template <int BITS>
__global__ void kv_pack_v_kernel(const uint8_t* __restrict__ codes, int B, int L, int Hkv,
                                 uint8_t* __restrict__ tiles) {
  constexpr int RB = kAttnD * BITS / 8;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (b, kvh, tile, dim)
  const long long total = (long long)B * Hkv * (L / 16) * kAttnD;
  if (idx >= total) return;
  const int dim = (int)(idx % kAttnD);
  long long rest = idx / kAttnD;
  const int tile = (int)(rest % (L / 16));
  rest /= (L / 16);
  const int kvh = (int)(rest % Hkv);
  const int b = (int)(rest / Hkv);
  uint32_t c[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint8_t byte = codes[(((size_t)b * L + tile * 16 + i) * Hkv + kvh) * RB + (BITS == 8 ? dim : dim / 2)];
    c[i] = BITS == 8 ? byte : ((dim & 1) ? (byte >> 4) : (byte & 15u));
  }
  if constexpr (BITS == 8) {
    uint4 v;
    v.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    v.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    v.z = c[8] | (c[9] << 8) | (c[10] << 16) | (c[11] << 24);
    v.w = c[12] | (c[13] << 8) | (c[14] << 16) | (c[15] << 24);
    reinterpret_cast<uint4*>(tiles)[idx] = v;
  } else {
    uint2 v;
    v.x = c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12) | (c[4] << 16) | (c[5] << 20) | (c[6] << 24) | (c[7] << 28);
    v.y = c[8] | (c[9] << 4) | (c[10] << 8) | (c[11] << 12) | (c[12] << 16) | (c[13] << 20) | (c[14] << 24) |
          (c[15] << 28);
    reinterpret_cast<uint2*>(tiles)[idx] = v;
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
  return cudaLaunchKernelEx(&cfg, kv_attn_tc_kernel<BITS, G>, P) == cudaSuccess ? TM_OK : TM_ERR_CUDA;
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
  if (B < 0 || Hq <= 0 || Hkv <= 0 || L < 0 || L % 16 != 0 || Hq % Hkv != 0 || D != kAttnD ||
      (bits != 4 && bits != 8))
    return TM_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return TM_ERR_UNSUPPORTED;
  if (split < 0 || split > max_split(G) || (split & (split - 1))) return TM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(out)) & 3u) return TM_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & (bits == 8 ? 15u : 7u) ||
      (reinterpret_cast<uintptr_t>(Q) & 7u))
    return TM_ERR_ALIGNMENT;
  if (B == 0) return TM_OK;
  int S = split;
  if (!S) {
    // enough CTAs to cover the SMs twice, each with at least 256 tokens
    const int sms = num_sms(0);
    S = 1;
    while (S < max_split(G) && B * Hkv * S < 2 * sms && L / (2 * S) >= 256) S *= 2;
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
    if (G == 8) r = attn_launch<8, 8>(P, B, S, st);
  } else {
    if (G == 1) r = attn_launch<4, 1>(P, B, S, st);
    if (G == 2) r = attn_launch<4, 2>(P, B, S, st);
    if (G == 4) r = attn_launch<4, 4>(P, B, S, st);
    if (G == 8) r = attn_launch<4, 8>(P, B, S, st);
  }
  if (r == TM_OK) set_launch_count(1);
  return r;
}

extern "C" tm_status tm_kv_pack_v(const uint8_t* codes, int B, int L, int Hkv, int bits, uint8_t* tiles,
                                  void* stream) {
  if (!codes || !tiles || B < 0 || L < 0 || Hkv <= 0 || L % 16 != 0 || (bits != 4 && bits != 8))
    return TM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(tiles) & (bits == 8 ? 15u : 7u)) return TM_ERR_ALIGNMENT;
  const long long total = (long long)B * Hkv * (L / 16) * kAttnD;
  if (total == 0) return TM_OK;
  const unsigned grid = (unsigned)((total + 255) / 256);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (bits == 8) {
    kv_pack_v_kernel<8><<<grid, 256, 0, st>>>(codes, B, L, Hkv, tiles);
  } else {
    kv_pack_v_kernel<4><<<grid, 256, 0, st>>>(codes, B, L, Hkv, tiles);
  }
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}
