/*
 * tm_w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 mixed-precision GEMM.
 *
 *   Y[M,N] = X[M,K] . dequant(W),   dequant(w)[k][n] = (q[k][n] - z[k/g][n]) * s[k/g][n]
 *
 * W is stored as unsigned 4-bit codes q (0..15), grouped along K in groups of
 * g weights, with one fp16 scale s and one 4-bit zero z per (group, column).
 * X and Y are fp16; products accumulate in fp32.
 *
 * Sources: the dequantisation rule is that of "LMDeploy Guide: Fast
 * Mixed-Precision LLM Inference Engine", section 3 ("Instruction-Level
 * Parallelism (ILP) for Zero-Overhead Dequantization"); groups run along K
 * with one scale per group ("LMDeploy, in depth", section "Quantization: AWQ
 * weights and KV cache"); the weights are repacked once, offline, into the
 * order the kernels consume so that no layout change happens at run time (the
 * guide, section 1 "Hardware-Aware Weight Packing").
 *
 * Conventions for every call:
 *   - Pointers named "device" must point to memory of the current CUDA device.
 *   - Kernels wait on barriers for at most about one second.  A wait that
 *     gives up (a GPU time-sliced away for longer, or a copy that never
 *     lands) cannot change the status the launching call already returned:
 *     it sets a sticky device bit instead, and the outputs of that launch are
 *     undefined (possibly stale) until tm_device_error reports the bit clear.
 *   - fp16 values travel as their 16-bit patterns (uint16_t) or as void*.
 *   - Nothing throws; every call returns a tm_status (or nothing).
 *   - Shapes: g in {64, 128}; K > 0 and K % g == 0; N > 0 and N % 16 == 0;
 *     M >= 0 (M == 0 is a no-op).
 */
#ifndef TM_W4A16_H
#define TM_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TM_OK = 0,
  TM_ERR_INVALID_ARG = 1,   /* null pointer, bad shape or group size */
  TM_ERR_ALIGNMENT = 2,     /* a pointer is not 16-byte aligned */
  TM_ERR_UNSUPPORTED = 3,   /* valid request this build does not serve (e.g. no sm_103a device) */
  TM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  TM_ERR_DEVICE_TIMEOUT = 5,/* a kernel gave up waiting on a barrier (reported by tm_device_error) */
  TM_ERR_BAD_CODE = 6,      /* a code or zero above 15 was passed to tm_pack_weights */
  TM_ERR_SCRATCH_LIMIT = 7  /* the request does not fit the static staging array of tm_w4a16_gemm_host_static */
} tm_status;

/* Opaque packed weights.  Owns one device allocation (codes, scales, zeros in
 * the kernels' order) on the device that was current at tm_pack_weights. */
typedef struct tm_packed tm_packed;

/* Optional launch settings for tm_w4a16_gemm_ex; zero fields mean "automatic". */
typedef struct {
  int path;    /* 0 auto, 1 decode kernel (mma.sync, M <= 64), 2 prefill kernel (tcgen05, W^T staged in
                  shared memory), 3 tensor-memory kernel (tcgen05, W^T dequantised into tensor memory) */
  int split_k; /* 0 auto, else number of CTAs (a thread-block cluster, 1..8) sharing one output tile along K */
  int tile_n;  /* 0 auto, else output columns per CTA (decode 64/128/256, prefill 256, tensor-memory 128) */
  int stages;  /* 0 auto, else pipeline depth in shared memory (decode 2..8, prefill 6, tensor-memory 2..16) */
  int warp_n;  /* decode only: 0 auto, else 16-column tiles per consumer warp (1, 2 or 4) */
  int tile_m;  /* tensor-memory path only: 0 auto, else rows of X per CTA (16, 32, 64, 128 or 256) */
} tm_gemm_config;

/* Human-readable name of a status (static string, never NULL). */
const char* tm_status_str(tm_status s);

/* Bytes of device memory tm_pack_weights allocates for a K x N layer with
 * group size g.  Writes *bytes; TM_ERR_INVALID_ARG on a bad shape. */
tm_status tm_packed_bytes(int K, int N, int g, size_t* bytes);

/*
 * Offline repack (the guide's section 1): reads the plain codes and scales
 * and writes them, once, in the fragment order the GEMM kernels load.
 *   q : device, uint8 [K][N] row-major, one code (0..15) per byte
 *   z : device, uint8 [K/g][N], one zero (0..15) per byte
 *   s : device, fp16 bits [K/g][N]
 *   out: receives a new handle; the caller frees it with tm_packed_free.
 * Synchronous: returns after the packing kernels finished on the current
 * device.  TM_ERR_BAD_CODE if any q or z is above 15 (no handle is returned).
 */
tm_status tm_pack_weights(const uint8_t* q, const uint8_t* z, const uint16_t* s, int K, int N, int g,
                          tm_packed** out);

/* Inverse of tm_pack_weights (device pointers with the same layouts as its
 * inputs; the caller owns them).  Synchronous.  pack -> unpack is bit-exact. */
tm_status tm_unpack_weights(const tm_packed* p, uint8_t* q, uint8_t* z, uint16_t* s);

/* K, N, g and the size of the device allocation of a handle (any out pointer may be NULL). */
tm_status tm_packed_info(const tm_packed* p, int* K, int* N, int* g, size_t* bytes);

/*
 * Round-to-nearest INT4 quantisation ("LMDeploy, in depth", section
 * "Quantization: AWQ weights and KV cache": naive RTN INT4 is the baseline the
 * pages compare AWQ against), producing exactly the inputs of tm_pack_weights.
 * For every group G of g rows along K and column n, in IEEE binary32 with
 * round-to-nearest-even at each step:
 *   lo = min(0, min w), hi = max(0, max w); r = hi - lo, or 15 if r == 0
 *   s[G][n] = fp16(r / 15), at least 2^-24 (the smallest positive fp16)
 *   z[G][n] = clamp(rint(-lo / s), 0, 15)
 *   q[k][n] = clamp(rint(w[k][n] / s) + z, 0, 15)
 * (the division per weight is computed as a multiply by 1/s and one fma
 * correction, which gives the quotient's integer rounding exactly, ties
 * included, for fp16 w and s)
 *   W : device, fp16 bits [K][N] row-major, 16-byte aligned
 *   q : device, uint8 [K][N] (one code per byte), 8-byte aligned
 *   z : device, uint8 [K/g][N], 8-byte aligned;  s: device, fp16 bits [K/g][N], 16-byte aligned
 * K % g == 0, N % 16 == 0, K/g <= 65535.  Asynchronous on `stream` (one launch,
 * no allocation); the caller owns every buffer.  TM_ERR_INVALID_ARG on a bad
 * shape or NULL pointer, TM_ERR_ALIGNMENT on a misaligned pointer.
 */
tm_status tm_quantize_rtn(const uint16_t* W, int K, int N, int g, uint8_t* q, uint8_t* z, uint16_t* s,
                          void* stream);

/*
 * Low-bit KV cache ("LMDeploy, in depth", section "Quantization: AWQ weights
 * and KV cache": int8 / int4 keys and values, quantised online,
 * asymmetrically, per head and per token).
 *
 * tm_kv_quantize: `rows` vectors of D fp16 values (one per (token, head),
 * D = 64, 128 or 256) -> codes, an fp16 scale and a uint8 zero per vector, by
 * the rule of tm_quantize_rtn with B = 2^bits - 1 in place of 15:
 *   lo = min(0, min x), hi = max(0, max x); r = hi - lo, or B if r == 0;
 *   s = fp16(r / B) (>= 2^-24); z = clamp(rint(-lo / s), 0, B);
 *   q = clamp(rint(x / s) + z, 0, B)          (IEEE binary32, ties to even)
 *   X     : device fp16 [rows][D], 4-byte aligned
 *   codes : device uint8 [rows][D] (bits 8) or [rows][D/2] (bits 4, even
 *           index in the low nibble); s: fp16 [rows]; z: uint8 [rows]
 * Asynchronous on `stream`, one launch.
 */
tm_status tm_kv_quantize(const uint16_t* X, long long rows, int D, int bits, uint8_t* codes, uint16_t* s,
                         uint8_t* z, void* stream);

/*
 * Value codes of the head-major cache, [B][Hkv][L][D*bits/8] with D = 128 (as
 * tm_kv_quantize writes them for vectors ordered (sequence, KV head, token)),
 * to the tiles tm_kv_decode_attention reads: [B][Hkv][L/16][16*D*bits/8],
 * each 16-token tile in MMA A-fragment order, 16-byte chunk (c, lane = 4 gr + t):
 * int8 -- 4 chunks, word k of chunk c holds the codes of dimension
 * 8(4c + k) + gr for tokens 2t, 2t+1, 2t+8, 2t+9 (a byte each); int4 -- 2
 * chunks, word k of chunk c belongs to MMA p = 4c + k, its nibbles 0..7 being
 * (token, dimension) (2t, A), (2t+8, A), (2t, B), (2t+8, B), (2t+1, A),
 * (2t+9, A), (2t+1, B), (2t+9, B) with A = 16p + gr, B = A + 8.  L % 16 == 0;
 * tiles 16-byte aligned.  Asynchronous on `stream`, one launch.
 */
tm_status tm_kv_pack_v(const uint8_t* codes, int B, int L, int Hkv, int bits, uint8_t* tiles, void* stream);

/*
 * Online append to the head-major cache: the new token of every (sequence b,
 * KV head) is quantised by the rule of tm_kv_quantize and written at position
 * pos[b] -- key codes, ks, kz, vs, vz in place and the value codes into the
 * 16-token tile of tm_kv_pack_v's layout (int4: the byte shared with token
 * pos +- 8 is read, modified and written).  Positions outside 0..L-1 are
 * ignored.  One token per sequence per call.
 *   Kn, Vn : device fp16 [B][Hkv][D], D = 128, 8-byte aligned
 *   pos    : device int32 [B]
 *   kc, ks, kz, vtiles, vs, vz: the cache of tm_kv_decode_attention (kc 4-byte,
 *            ks and vs 2-byte aligned), L % 16 == 0
 * Asynchronous on `stream`, one launch.
 */
tm_status tm_kv_append(const uint16_t* Kn, const uint16_t* Vn, const int* pos, int B, int Hkv, int L, int D, int bits,
                       uint8_t* kc, uint16_t* ks, uint8_t* kz, uint8_t* vtiles, uint16_t* vs, uint8_t* vz,
                       void* stream);

/*
 * Decode attention over a quantised KV cache, one query token per sequence,
 * on tensor cores (mma.m16n8k16 on the codes as exact fp16 integers):
 *   out[b][h] = sum_t p_t v~_t,  p = softmax_t(q[b][h] . k~_t / sqrt(D)),
 *   t < lengths[b], k~ = (qk - zk) sk, v~ = (qv - zv) sv, KV head h / (Hq/Hkv).
 * The cache is head-major (each KV head's tokens contiguous):
 *   Q      : device fp16 [B][Hq][D], D = 128; out: fp16 [B][Hq][D]
 *   kc     : key codes [B][Hkv][L][D*bits/8]
 *   vc     : value codes as tiles from tm_kv_pack_v
 *   ks, vs : fp16 and kz, vz uint8 per (token, head): [B][Hkv][L]
 *   Q, kc, vc, ks, vs, kz, vz 16-byte aligned (TM_ERR_ALIGNMENT otherwise)
 *   L      : cache capacity in tokens, a multiple of 16
 *   lengths: device int32 [B] (clamped to 0..L; 0 gives a zero output)
 *   split  : CTAs per (sequence, KV head) along the tokens (a cluster, 1..8
 *            (1..4 for 8 query heads per KV head), power of two; 0 =
 *            automatic); partial softmax states combine through distributed
 *            shared memory, no global workspace.
 * Hq / Hkv must be 1, 2, 4 or 8 (TM_ERR_UNSUPPORTED otherwise).  Scores and
 * softmax in fp32; the value weights p s_v are rounded once to fp16 for the
 * product.  Waits are bounded: a copy that never lands sets the device
 * timeout bit (tm_device_error).  Asynchronous on `stream`, one launch.
 */
tm_status tm_kv_decode_attention(const uint16_t* Q, const uint8_t* kc, const uint16_t* ks, const uint8_t* kz,
                                 const uint8_t* vc, const uint16_t* vs, const uint8_t* vz, const int* lengths,
                                 int B, int Hq, int Hkv, int L, int D, int bits, int split, uint16_t* out,
                                 void* stream);

/* Release a handle and its device memory (NULL is ignored). */
void tm_packed_free(tm_packed* p);

/*
 * The product.  X: device fp16 [M][K] row-major, 16-byte aligned.
 * Y: device fp16 [M][N] row-major, 16-byte aligned, written in full.
 * stream: a cudaStream_t (NULL = the legacy default stream).
 * Asynchronous on `stream`; no host synchronisation, no allocation.
 * M <= 32 runs the decode kernel (split-K mma.sync GEMV/skinny GEMM),
 * larger M the tcgen05 tensor-memory kernel (W^T dequantised into tensor
 * memory as the MMA's A operand).  Different calls may share a handle
 * concurrently: a call keeps no state outside its own launch.
 */
tm_status tm_w4a16_gemm(const void* X, const tm_packed* p, void* Y, int M, void* stream);

/*
 * Fused gate/up product of a Llama MLP: H = silu(X . W_gate) * (X . W_up)
 * in one launch, silu(x) = x / (1 + exp(-x)) in fp32 on the fp32 sums.
 * The packed weight holds both halves with N = 2 I columns interleaved in
 * blocks of 4 (our convention): columns 8b .. 8b+3 are gate columns
 * 4b .. 4b+3 and columns 8b+4 .. 8b+7 the matching up columns.
 *   H: device fp16 [M][N/2] row-major, 16-byte aligned; H[m][4b + i] pairs
 *      W columns 8b + i (gate) and 8b + 4 + i (up).
 * Same paths, planning and status codes as tm_w4a16_gemm_ex (cfg may be NULL);
 * path 2 (shared-memory prefill kernel) returns TM_ERR_UNSUPPORTED.
 */
tm_status tm_w4a16_gemm_silu_mul(const void* X, const tm_packed* p, void* H, int M, const tm_gemm_config* cfg,
                                 void* stream);

/* Most products one tm_w4a16_gemm_grouped call puts in one launch. */
#define TM_GROUP_MAX 4

/* One product of tm_w4a16_gemm_grouped. */
typedef struct {
  const void* X;      /* device fp16 [M][K] row-major, 16-byte aligned (K: the handle's) */
  const tm_packed* p; /* packed weights, K x N */
  void* Y;            /* device fp16 [M][N] (silu: [M][N/2]) row-major, 16-byte aligned, written in full */
  int silu;           /* 0: Y = X . W;  1: Y = silu(X . W_gate) * (X . W_up) as tm_w4a16_gemm_silu_mul */
} tm_gemm_problem;

/*
 * n independent products of the same M in ONE kernel launch (the decode
 * kernel, M <= 32): the launch's CTAs cover the column blocks of all n
 * products, so the weight stream of one product runs on while another's
 * last CTAs reduce and store, and the launch's start-up and tail are paid
 * once instead of n times.  The products are those of tm_w4a16_gemm /
 * tm_w4a16_gemm_silu_mul, bit for bit equal to them under the same launch
 * settings (tile_n, warp_n and the product's split as split_k: see
 * tm_gemm_plan_grouped).  The paper
 * has no counterpart to this call; it is a property of this library.
 *
 *   probs: host array of n products, 1 <= n <= TM_GROUP_MAX; every handle on
 *          the current device, all with the same group size g (K and N may
 *          differ).  No product may read what another writes: every Y must
 *          be disjoint from every X and from every other Y (checked on the
 *          address ranges: TM_ERR_INVALID_ARG).
 *   cfg:   NULL = automatic, else path 0 or 1 and the decode fields, applied
 *          to every product: tile_n 64 or 128, warp_n 0 or 1, stages, and
 *          split_k (every product split that many ways; automatic: each
 *          product split by its own K, see tm_gemm_plan_grouped).
 * M > 32 with automatic settings runs the n products one after another, as n
 * tm_w4a16_gemm calls would (n launches).  Asynchronous on `stream`; no
 * allocation.  M == 0 is a no-op.  Errors: TM_ERR_INVALID_ARG (NULL pointer,
 * n out of range, mixed group sizes, overlapping buffers, silu with
 * N % 8 != 0), TM_ERR_ALIGNMENT, TM_ERR_UNSUPPORTED (settings the decode
 * kernel does not serve), TM_ERR_CUDA.  tm_last_launch_count reports the
 * launches made.
 */
tm_status tm_w4a16_gemm_grouped(const tm_gemm_problem* probs, int n, int M, const tm_gemm_config* cfg, void* stream);

/* The settings tm_w4a16_gemm_grouped would use (all fields of *out filled
 * in; out->split_k is the cluster size of the launch) and, when `splits` is
 * not NULL, each product's split along K (splits[i], a power of two dividing
 * out->split_k; automatic settings split each product by its own K).  Only
 * X, p and silu of each problem are read.  With M > 32 and automatic
 * settings, *out is the first product's own plan and splits[i] each
 * product's own split. */
tm_status tm_gemm_plan_grouped(const tm_gemm_problem* probs, int n, int M, const tm_gemm_config* cfg,
                               tm_gemm_config* out, int* splits);

/* tm_w4a16_gemm with explicit launch settings (cfg may be NULL = automatic). */
tm_status tm_w4a16_gemm_ex(const void* X, const tm_packed* p, void* Y, int M, const tm_gemm_config* cfg,
                           void* stream);

/*
 * The product with X and Y in host memory, all asynchronous on `stream`:
 * X_host is copied into X_dev, the product (as tm_w4a16_gemm_ex) runs from
 * X_dev into Y_dev, and Y_dev is copied back into Y_host.  The caller
 * synchronises the stream before reading Y_host.
 *   X_host: fp16 [M][K] row-major; Y_host: fp16 [M][N] row-major.  Pinned
 *           (page-locked) host memory lets the copies run asynchronously;
 *           pageable memory is accepted, the copies then block the caller.
 *   X_dev, Y_dev: device buffers of at least M K and M N fp16, 16-byte aligned
 *           (owned by the caller, so that the call allocates nothing).
 * Arguments are checked and the launch planned before any copy is issued:
 * TM_ERR_INVALID_ARG / TM_ERR_ALIGNMENT / TM_ERR_UNSUPPORTED leave every
 * buffer untouched; TM_ERR_CUDA when a copy or the launch fails.
 */
tm_status tm_w4a16_gemm_host(const void* X_host, const tm_packed* p, void* Y_host, int M, void* X_dev, void* Y_dev,
                             const tm_gemm_config* cfg, void* stream);

/*
 * n products with host inputs and outputs, staged through one copy each way
 * (the form of a decode step: every layer's activations in, every result out):
 *   X_host holds X_0 .. X_{n-1} back to back, X_i fp16 [M[i]][K_i] row-major
 *   (K_i, N_i: the shape of p[i]); Y_host receives Y_0 .. Y_{n-1} the same way.
 *   X_dev, Y_dev: device staging buffers of at least sum M[i] K_i and
 *   sum M[i] N_i fp16, 16-byte aligned; every X_i and Y_i then starts on a
 *   32-byte boundary (K_i % 64 == 0, N_i % 16 == 0).
 * On `stream`: one host-to-device copy, the n products in order (automatic
 * plans), one device-to-host copy; asynchronous, the caller synchronises
 * before reading Y_host.  Consecutive products with the same M <= 32 and the
 * same g, up to TM_GROUP_MAX of them, share one launch as in
 * tm_w4a16_gemm_grouped (automatic settings); every other product runs as
 * tm_w4a16_gemm.  Every product is planned before the first copy: a rejected
 * argument leaves all buffers untouched.  M[i] == 0 skips product i.
 * tm_last_launch_count reports the kernels of all n.
 */
tm_status tm_w4a16_gemm_host_batch(int n, const tm_packed* const* p, const int* M, const void* X_host, void* Y_host,
                                   void* X_dev, void* Y_dev, void* stream);

/*
 * Bytes of the device array behind tm_w4a16_gemm_host_static.  Every device
 * on which the library is loaded reserves this much memory when the module
 * loads there, and keeps it until the process exits.
 */
#define TM_STATIC_STAGING_BYTES (8u << 20)

/*
 * tm_w4a16_gemm_host without caller-provided device buffers, for callers
 * that cannot allocate device memory when they need the product: a plug-in
 * whose host application has already reserved the device for its own memory
 * pool (cudaMalloc then fails, or eats into that pool), or a latency-critical
 * loop where cudaMalloc / cudaFree may block or synchronise the device.  The
 * paper has no counterpart to this call; it is a property of this library.
 *
 * X_host (fp16 [M][K]) is copied into a fixed __device__ array of
 * TM_STATIC_STAGING_BYTES bytes, the product runs as tm_w4a16_gemm_ex from
 * there into the same array (Y at the first 256-byte boundary after X), and
 * Y comes back into Y_host (fp16 [M][N]).  Asynchronous on `stream`; the
 * caller synchronises the stream before reading Y_host.  Pinned host memory
 * lets the copies run asynchronously; pageable memory makes them block.
 *
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.
 *
 * Every call on a device shares the one array, which keeps the last call's
 * contents (nothing in it has to start at zero: X is copied in whole and Y
 * written in whole).  Calls whose copies or kernels overlap on the GPU --
 * on different streams, or from different host threads without ordering --
 * race on it and corrupt each other's X and Y: issue them on one stream.
 *
 * Errors: TM_ERR_INVALID_ARG for NULL pointers, M < 0, or a handle packed on
 * another device than the current one; TM_ERR_SCRATCH_LIMIT when
 * round_up(2 M K, 256) + 2 M N exceeds TM_STATIC_STAGING_BYTES (nothing is
 * copied or launched); otherwise as tm_w4a16_gemm_host.  M == 0 is a no-op.
 */
tm_status tm_w4a16_gemm_host_static(const void* X_host, const tm_packed* p, void* Y_host, int M,
                                    const tm_gemm_config* cfg, void* stream);

/* The settings tm_w4a16_gemm would use for this handle and M (all fields filled in). */
tm_status tm_gemm_plan(const tm_packed* p, int M, const tm_gemm_config* cfg, tm_gemm_config* out);

/* Sticky device-side error bits of the current device, set by kernels that
 * gave up waiting (bit 0: barrier timeout).  Synchronises the device.
 * clear != 0 resets them.  Returns TM_ERR_DEVICE_TIMEOUT when bit 0 was set. */
tm_status tm_device_error(int clear, uint32_t* bits);

/* Self-test of the bounded barrier waits (failure detection without a fault):
 * launches one warp that waits on a barrier nothing arrives on; after about
 * one second the wait gives up, sets bit 0 and the kernel returns, leaving
 * the context usable.  Asynchronous on `stream`; read the outcome with
 * tm_device_error (expected: TM_ERR_DEVICE_TIMEOUT, bits == 1). */
tm_status tm_selftest_wait_timeout(void* stream);

/* Number of kernel launches the last tm_w4a16_gemm* call on this thread made (1 or 0). */
int tm_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TM_W4A16_H */
