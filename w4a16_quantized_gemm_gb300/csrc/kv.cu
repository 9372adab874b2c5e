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
//   q = clamp(rint(x / s) + z, 0, B)   (the division as fp16_quotient: a
//   reciprocal per vector and one fma correction, ties included)
// Codes: one byte each (int8) or two per byte, even index in the low nibble
// (int4); s fp16 and z uint8 per (token, head).
//
// Cache layout (ours; the pages' paged cache keeps each KV head's tokens
// together inside a block): head-major, so that the 16-token tiles of one
// (sequence, KV head) are contiguous --
//   key codes   [B][Hkv][L][D * bits / 8]   (as tm_kv_quantize writes them)
//   value codes [B][Hkv][L / 16][tile]      (tm_kv_pack_v re-lays each tile in
//                                           the MMA lane order)
//   ks, kz, vs, vz [B][Hkv][L]
//
// Attention, one query token per sequence, D = 128, G = Hq / Hkv query heads
// per KV head: a CTA takes one (sequence, KV head) and a slice of its tokens;
// a producer warp streams them through a ring of shared-memory slots of 112
// tokens (bulk copies completing on mbarriers), and each of 7 consumer warps
// takes one 16-token tile of every slot and keeps an online softmax per head;
// the warps' states combine in shared memory, then over the CTAs of a
// thread-block cluster through distributed shared memory (no global scratch),
// and rank 0 writes the output.
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
  for (int e = 0; e < EPL; ++e) c[e] = (uint32_t)fminf(fmaxf(rintf(fp16_quotient(v[e], sf, inv)) + zf, 0.f), kB);
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
// Seven compute warps and the producer: 8 warps of up to 128 registers, so
// that two CTAs share an SM (each of the SM's four schedulers holds 16K
// registers: 4 warps x 128; a ninth warp per CTA would leave one CTA per SM).
constexpr int kConsumers = 7;                    // warps that compute, one 16-token tile of a slot each
constexpr int kAttnThreads = 32 * (kConsumers + 1);  // + one producer warp
constexpr int kSlotTiles = kConsumers;           // 16-token tiles per ring slot
constexpr int kState = 2 + kAttnD;               // max, sum, 128 accumulators per query head
constexpr int kMaxSplit = 8;                     // CTAs per cluster along the tokens

__device__ uint32_t s_err_kv;

// One ring slot holds 7 consecutive 16-token tiles of one (sequence, KV
// head): key codes (rows of D * BITS / 8 bytes), value tiles, then ks, vs
// (fp16) and kz, vz (uint8) per token; each region sized for 7 tiles and
// filled from its start (the last slot of a CTA may hold fewer tiles).
template <int BITS>
struct KvSlot {
  static constexpr uint32_t kTile = 16 * kAttnD * BITS / 8;  // code bytes of one tile
  static constexpr uint32_t kK = 0, kV = kSlotTiles * kTile, kKs = 2 * kSlotTiles * kTile;
  static constexpr uint32_t kVs = kKs + 32 * kSlotTiles, kKz = kVs + 32 * kSlotTiles, kVz = kKz + 16 * kSlotTiles;
  static constexpr uint32_t kBytes = kVz + 16 * kSlotTiles;
  static constexpr int kDepth = BITS == 8 ? 3 : 6;  // ~90 KB: two CTAs per SM
  static constexpr uint32_t kRing = kDepth * kBytes;
  static constexpr uint32_t kCombine = (uint32_t)(kConsumers + kMaxSplit) * 8 * kState * 4;  // G <= 8
  static constexpr uint32_t kBarOff = kRing > kCombine ? kRing : kCombine;
  static constexpr uint32_t kSmem = kBarOff + 16 * kDepth + 16;  // full, empty barriers; abort flag
};

struct AttnParams {
  const __half* Q;     // [B][Hq][D]
  const uint8_t* kc;   // [B][Hkv][L][D * BITS / 8]
  const __half* ks;    // [B][Hkv][L]
  const uint8_t* kz;   // [B][Hkv][L]
  const uint8_t* vc;   // [B][Hkv][L / 16][16 * D * BITS / 8], lane order (tm_kv_pack_v)
  const __half* vs;
  const uint8_t* vz;
  const int* lengths;  // [B]
  __half* out;         // [B][Hq][D]
  int L, Hq, Hkv;
};

__device__ __forceinline__ bool kv_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(&s_err_kv, kErrTimeout);
      return false;
    }
  }
  return true;
}

// Combine the per-warp softmax states part[w][h][.] into one per CTA, then
// over the CTAs of the cluster through distributed shared memory into rank
// 0's cta[r][h][.], which writes out = acc / sum.
template <int G>
__device__ __forceinline__ void finish_attention(const float* part, float* cta, const AttnParams& P, int b, int kvh,
                                                 int S, int rank) {
  __syncthreads();
  if (S > 1) cluster_sync_all();  // every CTA of the cluster is past its loop before remote stores
  const uint32_t cta_base = smem_u32(cta);
  for (int e = threadIdx.x; e < G * kState; e += kAttnThreads) {
    const int h = e / kState, k = e % kState;
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) mx = fmaxf(mx, part[(w * G + h) * kState]);
    float v = 0.f;
    if (k == 0) {
      v = mx;
    } else {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float m = part[(w * G + h) * kState];
        const float s = m == -CUDART_INF_F ? 0.f : exp2f(m - mx);
        v = fmaf(part[(w * G + h) * kState + k], s, v);
      }
    }
    const int idx = (rank * G + h) * kState + k;
    if (S > 1) {
      st_dsmem_f32(map_shared_rank(cta_base + 4u * idx, 0u), v);
    } else {
      cta[idx] = v;
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
    for (int r = 0; r < S; ++r) mx = fmaxf(mx, cta[(r * G + h) * kState]);
    float num = 0.f, den = 0.f;
    if (mx != -CUDART_INF_F) {
      for (int r = 0; r < S; ++r) {
        const float m = cta[(r * G + h) * kState];
        if (m == -CUDART_INF_F) continue;
        const float w = exp2f(m - mx);
        den = fmaf(cta[(r * G + h) * kState + 1], w, den);
        num = fmaf(cta[(r * G + h) * kState + 2 + d], w, num);
      }
    }
    P.out[((size_t)b * P.Hq + kvh * G + h) * kAttnD + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
  }
}

// ------------------------------------------------ tensor-core attention -----
//
// Per consumer warp one 16-token tile of each slot, on mma.m16n8k16 with the
// tokens and the dimensions as the 16-row side and the (up to 8) query heads
// of the KV head as the 8 columns, so no accumulator is wasted:
//   scores^T [16 tokens x 8 heads] = K codes [16 x 128] . Q^T, 8 MMAs on the
//     codes in their raw fp16 form: the pattern of 1024 OR-ed with an int8
//     code is 1024 + c, an int4 code OR-ed in above the lowest nibble gives
//     1024 + 16 c (its query entry is then taken / 16, exact), so the MMA sums
//     Q . c plus a per-head constant (1024 times the query sum over the
//     dimensions without the factor 16, 64 times the rest), removed with the
//     zero point afterwards: score = s_k (Q . c - z_k sum Q) / sqrt(D), in
//     fp32, kept in units of log2 (the softmax uses powers of two).  The k
//     order is permuted the same way on K and Q so that a lane reads the 32
//     dimensions 32t .. 32t+31 it needs of a token with two (int8) or one
//     (int4) 16-byte loads: in slice sl the slots 2t, 2t+1, 2t+8, 2t+9 of lane
//     t hold dimensions 32t + 4sl + (0, 1, 2, 3) for int8 -- one byte-permute
//     per pair -- and 32t + 8(sl/2) + (0, 4, 1, 5) or (2, 6, 3, 7) for int4,
//     so that one mask-and-OR per pair takes the nibbles straight out of a
//     32-bit word.
//   out^T [128 dims x 8 heads] += V codes^T . P', 8 MMAs: P' = p s_v (rounded
//     once to fp16) is the score fragment transposed by two movmatrix; the
//     value tile holds, per lane, the codes of dimensions 8q + gr (q = 0..15)
//     for tokens 2t, 2t+1, 2t+8, 2t+9 in MMA A-fragment order (int4: one
//     32-bit word per MMA, the four pairs taken out by masks).  The value
//     zero point is removed once per head at the end (sum_t P'_t z_t).
// A lane (gr, t) owns query heads 2t and 2t+1 throughout: after the max over
// the tile's tokens (three shuffles) the online softmax is lane-local.

// Two int8 codes (bytes 2i, 2i+1 of w) -> two exact fp16 values.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t w, int i) {
  const uint32_t x = __byte_perm(w, 0x6464u, i == 0 ? 0x4140u : 0x4342u);  // (1024 + c0, 1024 + c1)
  return hsub2_u32(x, 0x64006400u);
}

// Raw form of two int8 key codes for the score MMA: (1024 + c0, 1024 + c1).
__device__ __forceinline__ uint32_t codes_raw(uint32_t w, int i) {
  return __byte_perm(w, 0x6464u, i == 0 ? 0x4140u : 0x4342u);
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// 2^x on the special-function unit (relative error about 2^-22; results below
// the normal range flush to zero, and 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BITS, int G>
__global__ void __maxnreg__(112) kv_attn_tc_kernel(const AttnParams P) {
  using SL = KvSlot<BITS>;
  constexpr int RB = kAttnD * BITS / 8;  // code bytes per (token, head)
  constexpr int NS = SL::kDepth;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x, b = bh / P.Hkv, kvh = bh % P.Hkv;
  const int S = gridDim.y, rank = blockIdx.y;
  const int n = max(0, min(P.lengths[b], P.L));
  const int chunk = ((n + S - 1) / S + 15) & ~15;  // whole 16-token tiles per CTA
  const int t_begin = min(n, rank * chunk), t_end = min(n, t_begin + chunk);
  const int nslots = (t_end - t_begin + 16 * kSlotTiles - 1) / (16 * kSlotTiles);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + SL::kBarOff, bar_empty = bar_full + 8 * NS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SL::kBarOff + 16 * NS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  float* part = reinterpret_cast<float*>(smem);  // overlays the ring after the loop
  float* cta = part + kConsumers * G * kState;

  if (warp == kConsumers) {
    // ---- producer: one lane streams the slots with bulk copies
    if (lane == 0) {
      const size_t seq = (size_t)bh * P.L;  // first token of this (sequence, KV head) in [B][Hkv][L]
      int issued = 0;
      for (int i = 0; i < nslots; ++i) {
        const int slot = i % NS;
        if (i >= NS && !kv_wait(bar_empty + 8 * slot, (uint32_t)(i / NS - 1) & 1u, abort_flag)) break;
        const int tok0 = t_begin + 16 * kSlotTiles * i;
        const int tiles = min(kSlotTiles, (t_end - tok0 + 15) / 16);
        const uint32_t dst = sbase + slot * SL::kBytes, bar = bar_full + 8 * slot;
        mbar_expect_tx(bar, (uint32_t)tiles * (2 * SL::kTile + 96));
        bulk_g2s(dst + SL::kK, P.kc + (seq + tok0) * RB, tiles * SL::kTile, bar);
        bulk_g2s(dst + SL::kV, P.vc + (seq + tok0) * RB, tiles * SL::kTile, bar);
        bulk_g2s(dst + SL::kKs, P.ks + seq + tok0, tiles * 32, bar);
        bulk_g2s(dst + SL::kVs, P.vs + seq + tok0, tiles * 32, bar);
        bulk_g2s(dst + SL::kKz, P.kz + seq + tok0, tiles * 16, bar);
        bulk_g2s(dst + SL::kVz, P.vz + seq + tok0, tiles * 16, bar);
        issued = i + 1;
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int k = max(0, issued - NS); k < issued; ++k) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(bar_full + 8 * (k % NS), (uint32_t)(k / NS) & 1u))
          if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(&s_err_kv, kErrTimeout);
            break;
          }
      }
    }
    __syncwarp();
    __syncthreads();  // the consumers have written `part`
    finish_attention<G>(part, cta, P, b, kvh, S, rank);
    return;
  }

  // ---- consumers
  const int gr = lane >> 2, t = lane & 3;
  // B fragments of Q^T (column gr = query head gr < G) in the permuted k order
  // (int4: odd dimensions / 16); for this lane's heads 2t, 2t+1 the sum of Q
  // over the dimensions and the constant the raw codes add to the MMA sum
  uint32_t qb[8][2];
  float qs0, qs1, off0, off1;
  {
    uint4 q4[4] = {};
    if (gr < G) {
      const uint4* qp = reinterpret_cast<const uint4*>(P.Q + ((size_t)b * P.Hq + kvh * G + gr) * kAttnD + 32 * t);
#pragma unroll
      for (int c = 0; c < 4; ++c) q4[c] = qp[c];
    }
    float qe = 0.f, qo = 0.f;  // sums over even and odd dimensions
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t wv[4] = {q4[c].x, q4[c].y, q4[c].z, q4[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
        qe += f.x;
        qo += f.y;
      }
      if constexpr (BITS == 8) {
        qb[2 * c][0] = wv[0];
        qb[2 * c][1] = wv[1];
        qb[2 * c + 1][0] = wv[2];
        qb[2 * c + 1][1] = wv[3];
      } else {
        // dimensions 8c + i of the lane's 32: slice 2c pairs (0, 4) and (1, 5),
        // slice 2c + 1 pairs (2, 6) and (3, 7); odd dimensions / 16 (exact)
        qb[2 * c][0] = __byte_perm(wv[0], wv[2], 0x5410u);
        qb[2 * c][1] = hmul2_u32(__byte_perm(wv[0], wv[2], 0x7632u), 0x2C002C00u);
        qb[2 * c + 1][0] = __byte_perm(wv[1], wv[3], 0x5410u);
        qb[2 * c + 1][1] = hmul2_u32(__byte_perm(wv[1], wv[3], 0x7632u), 0x2C002C00u);
      }
    }
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      qe += __shfl_xor_sync(0xffffffffu, qe, x);
      qo += __shfl_xor_sync(0xffffffffu, qo, x);
    }
    const float qsum = qe + qo;                                  // head gr
    const float off = 1024.f * qe + (BITS == 8 ? 1024.f : 64.f) * qo;
    qs0 = __shfl_sync(0xffffffffu, qsum, 8 * t);  // head 2t
    qs1 = __shfl_sync(0xffffffffu, qsum, 8 * t + 4);  // head 2t + 1
    off0 = __shfl_sync(0xffffffffu, off, 8 * t);
    off1 = __shfl_sync(0xffffffffu, off, 8 * t + 4);
  }
  const float scale = rsqrtf((float)kAttnD) * 1.4426950408889634f;  // 1 / sqrt(D), in log2 units

  // heads 2t, 2t+1: running max, and this lane's partial sums of p and p' z
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f;
  float o[8][4];  // out^T: dims 16p + gr (0, 1) and 16p + 8 + gr (2, 3); heads 2t (0, 2), 2t+1 (1, 3)
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[p][e] = 0.f;

  for (int i = 0; i < nslots; ++i) {
    const int slot = i % NS;
    if (!__all_sync(0xffffffffu, kv_wait(bar_full + 8 * slot, (uint32_t)(i / NS) & 1u, abort_flag))) break;
    const int t0 = t_begin + 16 * (kSlotTiles * i + warp);  // this warp's tile
    if (t0 < t_end) {
      const uint8_t* sp = smem + slot * SL::kBytes;
      // ---- scores^T: rows = tokens gr, gr + 8; columns = heads 2t, 2t + 1
      uint32_t wa[8], wb[8];  // code words of tokens gr and gr + 8
      {
        const uint8_t* ka = sp + SL::kK + (warp * 16 + gr) * RB;
        const uint8_t* kb = ka + 8 * RB;
        if constexpr (BITS == 8) {
          const uint4 alo = *reinterpret_cast<const uint4*>(ka + 32 * t);
          const uint4 ahi = *reinterpret_cast<const uint4*>(ka + 32 * t + 16);
          const uint4 blo = *reinterpret_cast<const uint4*>(kb + 32 * t);
          const uint4 bhi = *reinterpret_cast<const uint4*>(kb + 32 * t + 16);
          wa[0] = alo.x, wa[1] = alo.y, wa[2] = alo.z, wa[3] = alo.w;
          wa[4] = ahi.x, wa[5] = ahi.y, wa[6] = ahi.z, wa[7] = ahi.w;
          wb[0] = blo.x, wb[1] = blo.y, wb[2] = blo.z, wb[3] = blo.w;
          wb[4] = bhi.x, wb[5] = bhi.y, wb[6] = bhi.z, wb[7] = bhi.w;
        } else {
          const uint4 a = *reinterpret_cast<const uint4*>(ka + 16 * t);
          const uint4 c = *reinterpret_cast<const uint4*>(kb + 16 * t);
          wa[0] = a.x, wa[1] = a.y, wa[2] = a.z, wa[3] = a.w;
          wb[0] = c.x, wb[1] = c.y, wb[2] = c.z, wb[3] = c.w;
        }
      }
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};  // two chains over the slices
#pragma unroll
      for (int sl = 0; sl < 8; ++sl) {
        uint32_t a[4];
        if constexpr (BITS == 8) {
          a[0] = codes_raw(wa[sl], 0);
          a[1] = codes_raw(wb[sl], 0);
          a[2] = codes_raw(wa[sl], 1);
          a[3] = codes_raw(wb[sl], 1);
        } else {
          // word sl/2 holds dimensions 0..7 as nibbles 0..7: the low nibbles of
          // bytes 0 and 2 are dimensions 0 and 4, the high ones 1 and 5 (x 16);
          // shifted by a byte, 2 and 6, 3 and 7
          const uint32_t xa = (sl & 1) ? wa[sl >> 1] >> 8 : wa[sl >> 1];
          const uint32_t xb = (sl & 1) ? wb[sl >> 1] >> 8 : wb[sl >> 1];
          a[0] = lop3<0xEA>(xa, 0x000F000Fu, 0x64006400u);
          a[1] = lop3<0xEA>(xb, 0x000F000Fu, 0x64006400u);
          a[2] = lop3<0xEA>(xa, 0x00F000F0u, 0x64006400u);
          a[3] = lop3<0xEA>(xb, 0x00F000F0u, 0x64006400u);
        }
        mma_16816((sl & 1) ? d1 : d0, a, qb[sl][0], qb[sl][1]);
      }
      // per-token scales of tokens gr (index 0) and gr + 8 (index 1)
      const __half* ksp = reinterpret_cast<const __half*>(sp + SL::kKs) + warp * 16;
      const __half* vsp = reinterpret_cast<const __half*>(sp + SL::kVs) + warp * 16;
      const uint8_t* kzp = sp + SL::kKz + warp * 16;
      const uint8_t* vzp = sp + SL::kVz + warp * 16;
      const bool va = t0 + gr < t_end, vb = t0 + gr + 8 < t_end;
      const float ka_s = __half2float(ksp[gr]) * scale, kb_s = __half2float(ksp[gr + 8]) * scale;
      const float ka_z = (float)kzp[gr], kb_z = (float)kzp[gr + 8];
      // Q . c = raw sum - off; minus z_k sum Q
      const float s00 = va ? ka_s * (fmaf(-ka_z, qs0, d0[0] + d1[0]) - off0) : -CUDART_INF_F;  // token gr, head 2t
      const float s01 = va ? ka_s * (fmaf(-ka_z, qs1, d0[1] + d1[1]) - off1) : -CUDART_INF_F;  // token gr, head 2t+1
      const float s10 = vb ? kb_s * (fmaf(-kb_z, qs0, d0[2] + d1[2]) - off0) : -CUDART_INF_F;  // token gr+8, head 2t
      const float s11 = vb ? kb_s * (fmaf(-kb_z, qs1, d0[3] + d1[3]) - off1) : -CUDART_INF_F;  // token gr+8, head 2t+1
      float mt0 = fmaxf(s00, s10), mt1 = fmaxf(s01, s11);
#pragma unroll
      for (int x = 4; x < 32; x <<= 1) {
        mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, x));
        mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, x));
      }
      const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);  // finite: token t0 is valid
      const bool rescale = !__all_sync(0xffffffffu, mn0 == m0 && mn1 == m1);
      const float al0 = exp2_approx(m0 - mn0), al1 = exp2_approx(m1 - mn1);  // 0 on the first tile
      m0 = mn0;
      m1 = mn1;
      const float p00 = exp2_approx(s00 - mn0), p01 = exp2_approx(s01 - mn1), p10 = exp2_approx(s10 - mn0),
                  p11 = exp2_approx(s11 - mn1);
      l0 = fmaf(l0, al0, p00 + p10);
      l1 = fmaf(l1, al1, p01 + p11);
      // tokens past the length: p = 0, and their (unwritten) scales must not reach P'
      const float va_s = va ? __half2float(vsp[gr]) : 0.f, vb_s = vb ? __half2float(vsp[gr + 8]) : 0.f;
      const uint32_t pa = pack_half2(p00 * va_s, p01 * va_s);  // token gr: heads 2t, 2t+1
      const uint32_t pb = pack_half2(p10 * vb_s, p11 * vb_s);  // token gr + 8
      {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pa));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pb));
        const float za = (float)vzp[gr], zb = (float)vzp[gr + 8];
        z0 = fmaf(z0, al0, fmaf(fa.x, za, fb.x * zb));
        z1 = fmaf(z1, al1, fmaf(fa.y, za, fb.y * zb));
      }
      // B fragments of P' [16 tokens x 8 heads]: lane (gr, t) gets head gr at
      // tokens 2t, 2t+1 and 2t+8, 2t+9
      const uint32_t pb0 = movmatrix_trans(pa), pb1 = movmatrix_trans(pb);
      if (rescale) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          o[p][0] *= al0;
          o[p][1] *= al1;
          o[p][2] *= al0;
          o[p][3] *= al1;
        }
      }
      // ---- out^T += V^T P'
      constexpr int NC = BITS == 8 ? 4 : 2;
      uint32_t vw[4 * NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(sp + SL::kV + warp * SL::kTile + c * 512 + lane * 16);
        vw[4 * c] = u.x, vw[4 * c + 1] = u.y, vw[4 * c + 2] = u.z, vw[4 * c + 3] = u.w;
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        uint32_t a[4];
        if constexpr (BITS == 8) {
          a[0] = codes_to_half2(vw[2 * p], 0);
          a[1] = codes_to_half2(vw[2 * p + 1], 0);
          a[2] = codes_to_half2(vw[2 * p], 1);
          a[3] = codes_to_half2(vw[2 * p + 1], 1);
        } else {
          // nibbles: 0 / 4 tokens 2t / 2t+1 of dimension 16p + gr, 1 / 5 tokens
          // 2t+8 / 2t+9; shifted by a byte, the same for dimension 16p + 8 + gr
          const uint32_t w = vw[p], w8 = w >> 8;
          a[0] = hsub2_u32(lop3<0xEA>(w, 0x000F000Fu, 0x64006400u), 0x64006400u);
          a[1] = hsub2_u32(lop3<0xEA>(w8, 0x000F000Fu, 0x64006400u), 0x64006400u);
          a[2] = hfma2_u32(lop3<0xEA>(w, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
          a[3] = hfma2_u32(lop3<0xEA>(w8, 0x00F000F0u, 0x64006400u), 0x2C002C00u, 0xD400D400u);
        }
        mma_16816(o[p], a, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);  // the slot may be refilled
  }
  // partial sums over this lane's tokens -> per head (over gr)
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    z0 += __shfl_xor_sync(0xffffffffu, z0, x);
    z1 += __shfl_xor_sync(0xffffffffu, z1, x);
  }
  __syncthreads();  // every slot consumed and landed: `part` may overlay the ring
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = 2 * t + hh;
    if (h < G) {
      float* pw = part + (warp * G + h) * kState;
      if (gr == 0) {
        pw[0] = hh ? m1 : m0;
        pw[1] = hh ? l1 : l0;
      }
      const float zc = hh ? z1 : z0;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        pw[2 + 16 * p + gr] = o[p][hh] - zc;
        pw[2 + 16 * p + 8 + gr] = o[p][2 + hh] - zc;
      }
    }
  }
  finish_attention<G>(part, cta, P, b, kvh, S, rank);
}

// Value codes [B][Hkv][L][D * BITS / 8] -> tiles [B][Hkv][L / 16][16 * D *
// BITS / 8] in the kernel's A-fragment order, 16-byte chunk (c, lane = 4 gr +
// t): int8 -- 4 chunks; word k of chunk c holds the codes of dimension
// 8(4c + k) + gr for tokens 2t, 2t+1, 2t+8, 2t+9, one byte each; int4 -- 2
// chunks; word k of chunk c is MMA p = 4c + k, nibbles 0..7 = (token, dimension)
// (2t, A), (2t+8, A), (2t, B), (2t+8, B), (2t+1, A), (2t+9, A), (2t+1, B),
// (2t+9, B) with A = 16p + gr, B = A + 8.
template <int BITS>
__global__ void kv_pack_v_kernel(const uint8_t* __restrict__ codes, int B, int L, int Hkv,
                                 uint8_t* __restrict__ tiles) {
  constexpr int RB = kAttnD * BITS / 8;
  constexpr int NC = BITS == 8 ? 4 : 2;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // ((bh, tile), c, lane)
  const long long total = (long long)B * Hkv * (L / 16) * NC * 32;
  if (idx >= total) return;
  const int lane = (int)(idx & 31), c = (int)((idx >> 5) % NC);
  const long long tile = (idx >> 5) / NC;  // bh * L / 16 + tile in the sequence
  const int gr = lane >> 2, t = lane & 3;
  const uint8_t* src = codes + tile * 16 * RB;  // the tile's 16 token rows
  auto code = [&](int tok, int dim) -> uint32_t {
    if constexpr (BITS == 8) {
      return src[tok * RB + dim];
    } else {
      return (src[tok * RB + dim / 2] >> (4 * (dim & 1))) & 15u;
    }
  };
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (BITS == 8) {
      const int dim = 8 * (4 * c + k) + gr;
      w[k] = code(2 * t, dim) | (code(2 * t + 1, dim) << 8) | (code(2 * t + 8, dim) << 16) |
             (code(2 * t + 9, dim) << 24);
    } else {
      // word p = 4c + k: nibbles 0, 4 = tokens 2t, 2t+1 of dimension 16p + gr;
      // 1, 5 = tokens 2t+8, 2t+9; 2, 6 and 3, 7 the same for dimension 16p + 8 + gr
      const int p = 4 * c + k, da = 16 * p + gr, db = da + 8;
      w[k] = code(2 * t, da) | (code(2 * t + 8, da) << 4) | (code(2 * t, db) << 8) | (code(2 * t + 8, db) << 12) |
             (code(2 * t + 1, da) << 16) | (code(2 * t + 9, da) << 20) | (code(2 * t + 1, db) << 24) |
             (code(2 * t + 9, db) << 28);
    }
  }
  reinterpret_cast<uint4*>(tiles)[idx] = make_uint4(w[0], w[1], w[2], w[3]);
}

// Online append: the new token of every (sequence, KV head) -- one warp each,
// lane l holding dimensions 4l .. 4l+3 -- quantised by the rule above and
// written at position pos[b] of the head-major cache: key codes, scales and
// zeros in place, the value codes into their bytes (int8) or nibbles (int4,
// read-modify-write of the byte shared with token pos +- 8) of the 16-token
// tile.  One token per sequence per launch, so no two lanes touch one byte.
template <int BITS>
__global__ void __launch_bounds__(128) kv_append_kernel(const __half* __restrict__ Kn, const __half* __restrict__ Vn,
                                                         const int* __restrict__ pos, int B, int Hkv, int L,
                                                         uint8_t* __restrict__ kc, __half* __restrict__ ks,
                                                         uint8_t* __restrict__ kz, uint8_t* __restrict__ vt,
                                                         __half* __restrict__ vs, uint8_t* __restrict__ vz) {
  constexpr int RB = kAttnD * BITS / 8;
  const int bh = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (bh >= B * Hkv) return;
  const int b = bh / Hkv;
  const int p = pos[b];
  if (p < 0 || p >= L) return;  // outside the cache: ignored
  const size_t row = (size_t)bh * L + p;
  constexpr float kB = (float)((1 << BITS) - 1);
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint2 raw = *reinterpret_cast<const uint2*>((which ? Vn : Kn) + (size_t)bh * kAttnD + 4 * lane);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    const float v[4] = {f0.x, f0.y, f1.x, f1.y};
    float lo = fminf(fminf(fminf(0.f, v[0]), fminf(v[1], v[2])), v[3]);
    float hi = fmaxf(fmaxf(fmaxf(0.f, v[0]), fmaxf(v[1], v[2])), v[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    float r = hi - lo;
    if (r == 0.f) r = kB;
    __half sh = __float2half_rn(__fdiv_rn(r, kB));
    const __half tiny = __ushort_as_half((unsigned short)1);  // 2^-24
    if (__half2float(sh) < __half2float(tiny)) sh = tiny;
    const float sf = __half2float(sh);
    const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), kB);
    const float inv = __fdiv_rn(1.f, sf);
    uint32_t c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] = (uint32_t)fminf(fmaxf(rintf(fp16_quotient(v[e], sf, inv)) + zf, 0.f), kB);
    if (which == 0) {
      if constexpr (BITS == 8) {
        *reinterpret_cast<uint32_t*>(kc + row * RB + 4 * lane) = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      } else {
        *reinterpret_cast<uint16_t*>(kc + row * RB + 2 * lane) = (uint16_t)(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
      }
      if (lane == 0) {
        ks[row] = sh;
        kz[row] = (uint8_t)zf;
      }
    } else {
      uint8_t* tile = vt + ((size_t)bh * (L / 16) + p / 16) * (16 * RB);
      const int tau = p & 15, t = (tau & 7) >> 1;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 4 * lane + e;
        if constexpr (BITS == 8) {
          const int q8 = d >> 3, gr = d & 7;
          tile[(q8 >> 2) * 512 + (4 * gr + t) * 16 + 4 * (q8 & 3) + (tau & 1) + 2 * (tau >> 3)] = (uint8_t)c[e];
        } else {
          const int pm = d >> 4, rr = d & 15, gr = rr & 7;
          const int nib = (tau >> 3) + 2 * (rr >> 3) + 4 * (tau & 1);
          uint8_t* byte = tile + (pm >> 2) * 512 + (4 * gr + t) * 16 + 4 * (pm & 3) + (nib >> 1);
          *byte = (nib & 1) ? (uint8_t)((*byte & 0x0Fu) | (c[e] << 4)) : (uint8_t)((*byte & 0xF0u) | c[e]);
        }
      }
      if (lane == 0) {
        vs[row] = sh;
        vz[row] = (uint8_t)zf;
      }
    }
  }
}

// Launch with S CTAs per (sequence, KV head) along the tokens; S = 0 picks S:
// split the tokens while the grid still fits in one wave of resident CTAs (the
// kernel's occupancy, registers included) and every CTA keeps at least four
// slots of tokens.
template <int BITS, int G>
tm_status attn_launch(const AttnParams& P, int B, int S, cudaStream_t stream) {
  constexpr uint32_t smem = KvSlot<BITS>::kSmem;
  static std::atomic<unsigned long long> attr_set{0};  // one bit per device
  if (!smem_attr_once(attr_set, (const void*)kv_attn_tc_kernel<BITS, G>, (int)smem)) return TM_ERR_CUDA;
  if (!S) {
    const int device = current_device();
    if (device < 0 || device >= 64) return TM_ERR_CUDA;
    static std::atomic<int> per_sm_cache[64];  // resident CTAs per SM, per device (0 = not yet queried)
    int per_sm = per_sm_cache[device].load();
    if (per_sm == 0) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_attn_tc_kernel<BITS, G>, kAttnThreads, smem) !=
              cudaSuccess ||
          per_sm < 1)
        return TM_ERR_CUDA;
      per_sm_cache[device].store(per_sm);
    }
    const long long slots = (long long)num_sms(device) * per_sm;
    S = 1;
    while (S < kMaxSplit && (long long)B * P.Hkv * S * 2 <= slots && P.L / (2 * S) >= 4 * 16 * kSlotTiles) S *= 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * P.Hkv), (unsigned)S, 1);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
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

cudaError_t kv_error_bits(uint32_t* bits, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, s_err_kv, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(s_err_kv, &zero, sizeof(zero));
  }
  *bits = v;
  return e;
}

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
  if (split < 0 || split > kMaxSplit || (split & (split - 1))) return TM_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(kc) |
                        reinterpret_cast<uintptr_t>(ks) | reinterpret_cast<uintptr_t>(kz) |
                        reinterpret_cast<uintptr_t>(vc) | reinterpret_cast<uintptr_t>(vs) |
                        reinterpret_cast<uintptr_t>(vz);
  if ((a16 & 15u) || (reinterpret_cast<uintptr_t>(out) & 1u)) return TM_ERR_ALIGNMENT;
  if (B == 0) return TM_OK;
  const int S = split;
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
  if (reinterpret_cast<uintptr_t>(tiles) & 15u) return TM_ERR_ALIGNMENT;
  const long long total = (long long)B * Hkv * (L / 16) * (bits == 8 ? 4 : 2) * 32;
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

extern "C" tm_status tm_kv_append(const uint16_t* Kn, const uint16_t* Vn, const int* pos, int B, int Hkv, int L, int D,
                                  int bits, uint8_t* kc, uint16_t* ks, uint8_t* kz, uint8_t* vtiles, uint16_t* vs,
                                  uint8_t* vz, void* stream) {
  if (!Kn || !Vn || !pos || !kc || !ks || !kz || !vtiles || !vs || !vz) return TM_ERR_INVALID_ARG;
  if (B < 0 || Hkv <= 0 || L <= 0 || L % 16 != 0 || D != kAttnD || (bits != 4 && bits != 8))
    return TM_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(Kn) | reinterpret_cast<uintptr_t>(Vn)) & 7u) ||
      (reinterpret_cast<uintptr_t>(kc) & 3u) || ((reinterpret_cast<uintptr_t>(ks) | reinterpret_cast<uintptr_t>(vs)) & 1u))
    return TM_ERR_ALIGNMENT;
  if (B == 0) return TM_OK;
  const unsigned grid = (unsigned)((B * Hkv + 3) / 4);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto* Kh = reinterpret_cast<const __half*>(Kn);
  auto* Vh = reinterpret_cast<const __half*>(Vn);
  if (bits == 8) {
    kv_append_kernel<8><<<grid, 128, 0, st>>>(Kh, Vh, pos, B, Hkv, L, kc, reinterpret_cast<__half*>(ks), kz, vtiles,
                                              reinterpret_cast<__half*>(vs), vz);
  } else {
    kv_append_kernel<4><<<grid, 128, 0, st>>>(Kh, Vh, pos, B, Hkv, L, kc, reinterpret_cast<__half*>(ks), kz, vtiles,
                                              reinterpret_cast<__half*>(vs), vz);
  }
  if (cudaGetLastError() != cudaSuccess) return TM_ERR_CUDA;
  set_launch_count(1);
  return TM_OK;
}
