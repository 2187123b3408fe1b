// sm_103a OjaKV-style reconstruction-error scores on the 5th-generation
// tensor cores (tcgen05 + TMA + TMEM).
//
// "OjaKV: Context-Aware Online Low-Rank KV Cache Compression" (deep notes of
// the ACL 2026 Findings paper), method details, error-based token
// selection: with r_t = k_t - U U^T k_t the part of key t that the low-rank
// basis U misses,
//     e_t = (1/M) sum over the M rows q of the recent query window of |q . r_t| / sqrt(d),
// and the tokens with the largest e_t stay at full rank.
//
// U U^T is symmetric, so q . r_t = (P q) . k_t with P = I - U U^T, for any U.
// The work therefore splits into
//  1. k_oja_project: P q for the M query rows of every head, in fp32 (CUDA
//     cores; M x d x r per head, tiny next to the cache), stored as a pair of
//     bf16 operands hi + lo with hi = bf16(Pq) and lo = bf16(Pq - hi), so
//     that hi + lo holds Pq to about 2^-17 relative;
//  2. k_oja_scores: a dense contraction of every key against the 2M operand
//     rows -- D[t][m] = k_t . hi_m + k_t . lo_m -- on tcgen05.mma (kind::f16,
//     bf16 x bf16 -> fp32 in TMEM), then e_t = scale * sum_m |D[t][m]|.
//     Keys are bf16 and exact in the MMA, so the only rounding beyond fp32
//     accumulation is the split's 2^-17.
//
// k_oja_scores is a persistent, warp-specialised kernel, one CTA per SM:
//  * warp 0 (one thread): TMA producer. A tile is 128 tokens x 128 dims
//    (32 KB) loaded as two 128-byte-swizzled boxes of 64 dims into a ring of
//    shared-memory stages (full/empty mbarriers). When the head changes, it
//    also loads that head's 2 x M operand rows (after the MMAs of the
//    previous head have drained).
//  * warp 1: allocates the TMEM accumulators (two buffers); its lane 0
//    issues the MMAs -- M_mma = 128 tokens on the TMEM lanes, 8 K-steps of
//    16 dims, each one MMA with N_mma = 2M operand rows (hi and lo stacked,
//    M <= 128) or two with N_mma = M accumulating hi and lo together
//    (M > 128) -- and commits them to the stage's empty barrier and the
//    buffer's full barrier. An MMA costs about the same issue time for any
//    N up to 128, so fewer, wider MMAs per tile are what keeps pace with HBM.
//  * warps 2-9: epilogue, two groups of 4 warps when M is a multiple of 64
//    (else warps 2-5 alone). The warp with rank w (= warp id mod 4) owns
//    TMEM lanes 32w..32w+31, i.e. one token per thread: it reads its half of
//    the token's accumulator row (tcgen05.ld 32x32b, 64 columns per wait),
//    adds the hi and lo halves of each query column and sums their absolute
//    values in column order; the second group's partial sum is added to the
//    first's (through shared memory), which scales and stores e_t.
// Every tile of 128 tokens costs 8 MMAs of 128 x 2M x 16 against 32 KB read
// from HBM (2 x 2M flop per key byte, against a bf16 ridge near 280).
//
// Every mbarrier wait is bounded (1 s of %globaltimer). On a timeout the
// kernel sets MKV_DEV_TIMEOUT, every role leaves its loop, the producer
// waits (bounded) for its own copies in flight, the MMA thread waits for its
// MMAs to complete, and the TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "mkv_device.cuh"
#include "mkv_internal.h"

namespace mkv {
namespace {

using namespace dev;

constexpr int kTok = 128;                    // tokens per tile: the MMA's M, the TMEM lanes
constexpr int kHalfBytes = kTok * 128;       // one 64-dim box of a tile: 128 rows x 128 B
constexpr int kTileBytes = 2 * kHalfBytes;   // 32 KB
constexpr int kMaxStages = 6;
constexpr int kOjaThreads = 320;             // producer warp, MMA warp, 8 epilogue warps
constexpr int kProjThreads = 256;
constexpr uint64_t kOjaWaitNs = 1000000000ull;
constexpr int kSmemBudget = 227 * 1024;

// ------------------------------------------------------ 1: P q, hi + lo --

// Item = (head, block of `rows` query rows: 64, 32 or 16, the largest that
// divides n_query); the block has rows / 8 warps. Shared memory holds q as
// fp32 rows of stride 132, U [d, r] with its columns padded with zeros to rp
// = r rounded up to 4 and a row stride of 4 x odd words, and y = U^T q as rows
// of stride rp. Every shared load is a 16-byte vector and each thread keeps an
// 8 x 4 tile of sums in registers:
//   y[m][j] = sum_i q[m][i] U[i][j]   (i in order; 8 rows x 4 adjacent columns)
//   p[m][i] = q[m][i] - sum_j U[i][j] y[m][j]   (j in order; 8 rows x dims
//             lane + 32c, c < 4, so that a warp's U rows are consecutive)
// and writes hi = bf16(p), lo = bf16(p - hi) (the difference is exact). The
// zero padding adds fma(0, 0, s) terms, which leave every sum unchanged.
constexpr int kProjBlock = 8;     // rows per thread
constexpr int kProjQStride = 132; // fp32 words per staged q row

__host__ __device__ constexpr int proj_rank_pad(int rank) { return (rank + 3) & ~3; }
// a row stride of 4 x odd words: the 8 lanes of a quarter warp reading 16
// bytes from 8 consecutive rows hit 32 distinct banks
__host__ __device__ constexpr int proj_u_stride(int rank)
{
    return (proj_rank_pad(rank) / 4) % 2 == 1 ? proj_rank_pad(rank) : proj_rank_pad(rank) + 4;
}

__global__ void __launch_bounds__(kProjThreads)
k_oja_project(const __nv_bfloat16 *__restrict__ Q, const float *__restrict__ U, int n_query, int rank, int rows,
              int64_t n_items, __nv_bfloat16 *__restrict__ qhl)
{
    extern __shared__ __align__(16) float sm[];
    const int rp = proj_rank_pad(rank), us = proj_u_stride(rank);
    float *sq = sm;                          // [rows][132]
    float *sU = sq + rows * kProjQStride;    // [128][us]
    float *sy = sU + kHeadDim * us;          // [rows][rp]
    const int blocks = n_query / rows, nthr = (int)blockDim.x, tid = (int)threadIdx.x;
    const int n4 = kHeadDim * rank / 4;      // float4s of one head's basis
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int64_t head = item / blocks;
        const int m0 = (int)(item - head * blocks) * rows;
        const float4 *U4 = reinterpret_cast<const float4 *>(U + head * kHeadDim * rank);
        for (int base = 0; base < n4; base += nthr * 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int o = base + u * nthr + tid;
                if (o < n4) v[u] = __ldg(U4 + o);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int o = base + u * nthr + tid;
                if (o < n4) {
                    // element e = 4o + c sits at row e / rank, column e % rank
                    int i = (4 * o) / rank, j = 4 * o - i * rank;
                    sU[i * us + j] = v[u].x;
                    if (++j == rank) j = 0, ++i;
                    sU[i * us + j] = v[u].y;
                    if (++j == rank) j = 0, ++i;
                    sU[i * us + j] = v[u].z;
                    if (++j == rank) j = 0, ++i;
                    sU[i * us + j] = v[u].w;
                }
            }
        }
        for (int o = tid; o < kHeadDim * (rp - rank); o += nthr)  // zero the padding columns
            sU[(o / (rp - rank)) * us + rank + o % (rp - rank)] = 0.f;
        const uint4 *Q4 = reinterpret_cast<const uint4 *>(Q + ((size_t)head * n_query + m0) * kHeadDim);
        for (int o = tid; o < rows * kHeadDim / 8; o += nthr) {
            float f[8];
            bf16x8_to_f32(__ldg(Q4 + o), f);
            float4 *dst = reinterpret_cast<float4 *>(sq + (o >> 4) * kProjQStride + 8 * (o & 15));
            dst[0] = make_float4(f[0], f[1], f[2], f[3]);
            dst[1] = make_float4(f[4], f[5], f[6], f[7]);
        }
        __syncthreads();
        // y: (rows / 8) x (rp / 4) tiles
        for (int o = tid; o < (rows / kProjBlock) * (rp / 4); o += nthr) {
            const int mg = o / (rp / 4), j0 = 4 * (o - mg * (rp / 4));
            const float *q0 = sq + mg * kProjBlock * kProjQStride;
            float acc[kProjBlock][4];
#pragma unroll
            for (int r = 0; r < kProjBlock; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
            for (int i = 0; i < kHeadDim; i += 4) {
                float4 u[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) u[c] = *reinterpret_cast<const float4 *>(sU + (i + c) * us + j0);
#pragma unroll
                for (int r = 0; r < kProjBlock; ++r) {
                    const float4 qv = *reinterpret_cast<const float4 *>(q0 + r * kProjQStride + i);
                    const float qs[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[r][0] = fmaf(qs[c], u[c].x, acc[r][0]);
                        acc[r][1] = fmaf(qs[c], u[c].y, acc[r][1]);
                        acc[r][2] = fmaf(qs[c], u[c].z, acc[r][2]);
                        acc[r][3] = fmaf(qs[c], u[c].w, acc[r][3]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kProjBlock; ++r)
                *reinterpret_cast<float4 *>(sy + (mg * kProjBlock + r) * rp + j0) =
                    make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
        __syncthreads();
        // p: (rows / 8) x 32 tiles, one warp per 8 rows
        for (int o = tid; o < (rows / kProjBlock) * 32; o += nthr) {
            const int mg = o >> 5, lane = o & 31;
            const float *y0 = sy + mg * kProjBlock * rp;
            float acc[kProjBlock][4];
#pragma unroll
            for (int r = 0; r < kProjBlock; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
            for (int j = 0; j < rp; j += 4) {
                float4 u[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) u[c] = *reinterpret_cast<const float4 *>(sU + (lane + 32 * c) * us + j);
#pragma unroll
                for (int r = 0; r < kProjBlock; ++r) {
                    const float4 yv = *reinterpret_cast<const float4 *>(y0 + r * rp + j);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[r][c] = fmaf(u[c].x, yv.x, acc[r][c]);
                        acc[r][c] = fmaf(u[c].y, yv.y, acc[r][c]);
                        acc[r][c] = fmaf(u[c].z, yv.z, acc[r][c]);
                        acc[r][c] = fmaf(u[c].w, yv.w, acc[r][c]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kProjBlock; ++r) {
                const int m = mg * kProjBlock + r;
                const size_t row = (size_t)head * 2 * n_query + m0 + m;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int i = lane + 32 * c;
                    const float pv = sq[m * kProjQStride + i] - acc[r][c];
                    const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(pv - __bfloat162float(hi));
                    qhl[row * kHeadDim + i] = hi;
                    qhl[(row + n_query) * kHeadDim + i] = lo;
                }
            }
        }
        __syncthreads();  // shared memory is reused by the next item
    }
}

// ----------------------------------------------- 2: tcgen05 contraction --

__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint64_t *b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}

__device__ __forceinline__ void bar_expect(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}

// Bounded wait for phase `parity` of b. On timeout: flag, raise the CTA's
// abort flag, return false. An abortable wait also returns false as soon as
// another role raised the abort flag.
__device__ __forceinline__ bool bar_wait(uint64_t *b, uint32_t parity, uint32_t *status, volatile uint32_t *abort_flag,
                                         bool abortable)
{
    const uint32_t a = saddr(b);
    const uint64_t t0 = global_ns();
    for (uint32_t spin = 0;; ++spin) {
        uint32_t done;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(a), "r"(parity)
                     : "memory");
        if (done) return true;
        if ((spin & 63u) == 63u) {
            if (abortable && *abort_flag) return false;
            if (global_ns() - t0 > kOjaWaitNs) {
                atomicOr(status, MKV_DEV_TIMEOUT);
                *abort_flag = 1u;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *b)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(saddr(b))
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout TMA writes: rows of 128 B, 8-row groups 1024 B apart
// (stride byte offset), leading byte offset unused for this layout,
// descriptor version 1, layout type 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTok >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *b)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(b))
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// Query columns [c0, c0 + cw) of this thread's lane (cw a multiple of 16),
// read 64 at a time per wait. Stacked: the hi and lo partial dot products
// sit n columns apart and are added first; either way the absolute values
// are added in column order.
__device__ __forceinline__ float tmem_abs_sum(uint32_t taddr, uint32_t n, bool stacked, int c0, int cw)
{
    float s = 0.f;
    for (int c = c0; c < c0 + cw; c += 64) {
        const int nb = min(64, c0 + cw - c);
        uint32_t h[4][16], l[4][16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (16 * k < nb) {
                tmem_ld16(taddr + (uint32_t)(c + 16 * k), h[k]);
                if (stacked) tmem_ld16(taddr + n + (uint32_t)(c + 16 * k), l[k]);
            }
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (16 * k < nb) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x = __uint_as_float(h[k][i]);
                    if (stacked) x += __uint_as_float(l[k][i]);
                    s += fabsf(x);
                }
            }
        }
    }
    return s;
}

struct TileWalk {
    int64_t first, last;  // this CTA's tile range [first, last)
    int tph;              // tiles per head
};

__device__ __forceinline__ TileWalk tile_range(int64_t n_heads, int t_max)
{
    TileWalk w;
    w.tph = (t_max + kTok - 1) / kTok;
    const int64_t total = n_heads * w.tph;
    w.first = total * blockIdx.x / gridDim.x;
    w.last = total * (blockIdx.x + 1) / gridDim.x;
    return w;
}

__global__ void __launch_bounds__(kOjaThreads, 1)
k_oja_scores(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
             const int32_t *__restrict__ seq_lens, int heads, int t_max, int64_t n_heads, int n_query, int stages,
             uint32_t tmem_cols, float scale, float *__restrict__ S, uint32_t *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *kring = smem;                              // stages x 32 KB
    uint8_t *qbuf = smem + (size_t)stages * kTileBytes;  // [dims 0-63, 64-127][hi, lo][n_query rows x 128 B]
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], qfull, qempty, tfull[2], tempty[2], pready[2],
        drain;
    __shared__ float part[2][kTok];  // the second epilogue group's partial sums, per accumulator buffer
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile uint32_t abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t q_block = (uint32_t)n_query * 128u;  // bytes of one [half][split] block of operand rows
    const bool stacked = 2 * n_query <= 256;
    const int acc_cols = stacked ? 2 * n_query : n_query;  // fp32 columns of one accumulator
    // epilogue groups of 4 warps (one per TMEM lane quadrant), each summing
    // an equal share of the query columns: two when the share is a multiple
    // of 32 columns
    const int groups = n_query % 64 == 0 ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], 1);
        }
        bar_init(&qfull, 1);
        bar_init(&qempty, 1);
        for (int b = 0; b < 2; ++b) {
            bar_init(&tfull[b], 1);
            bar_init(&tempty[b], 4 * groups);
            bar_init(&pready[b], 4);
        }
        bar_init(&drain, 1);
        abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base_sh)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_base_sh;
    const TileWalk walk = tile_range(n_heads, t_max);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer --
            uint32_t seq = 0, qseq = 0;
            uint32_t last_parity[kMaxStages];
            int64_t cur = -1;
            for (int64_t tile = walk.first; tile < walk.last; ++tile) {
                const int64_t head = tile / walk.tph;
                const int t0 = (int)(tile - head * walk.tph) * kTok;
                if (t0 >= head_len(seq_lens, head, heads, t_max, status, false)) continue;
                if (head != cur) {
                    if (qseq > 0 && !bar_wait(&qempty, (qseq - 1) & 1u, status, &abort_flag, true)) break;
                    bar_expect(&qfull, 4u * q_block);
                    for (int split = 0; split < 2; ++split)
                        for (int half = 0; half < 2; ++half)
                            tma_load_2d(qbuf + (half * 2 + split) * q_block, &tmap_q, half * 64,
                                        (int)((head * 2 + split) * n_query), &qfull);
                    ++qseq;
                    cur = head;
                }
                const int s = (int)(seq % (uint32_t)stages);
                if (seq >= (uint32_t)stages &&
                    !bar_wait(&empty[s], ((seq / stages) - 1) & 1u, status, &abort_flag, true))
                    break;
                bar_expect(&full[s], (uint32_t)kTileBytes);
                const int row = (int)(head * t_max + t0);
                tma_load_2d(kring + (size_t)s * kTileBytes, &tmap_k, 0, row, &full[s]);
                tma_load_2d(kring + (size_t)s * kTileBytes + kHalfBytes, &tmap_k, 64, row, &full[s]);
                last_parity[s] = (seq / stages) & 1u;
                ++seq;
            }
            // Every copy issued lands before the CTA may exit (bounded; after
            // a normal run these phases are long complete).
            const uint32_t issued = seq < (uint32_t)stages ? seq : (uint32_t)stages;
            for (uint32_t s = 0; s < issued; ++s) bar_wait(&full[s], last_parity[s], status, &abort_flag, false);
            if (qseq > 0) bar_wait(&qfull, (qseq - 1) & 1u, status, &abort_flag, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer --
            // Descriptors of stage 0's first K-step and of the operand rows;
            // every other one differs by an address offset (in 16-byte units,
            // the low field of the descriptor). Operand rows sit in shared
            // memory as [dims 0-63, 64-127][hi, lo][n_query rows x 128 B], so
            // hi and lo of one half are 2M contiguous rows: one N = 2M
            // operand when that fits an MMA (M <= 128), else two of N = M.
            const uint32_t idesc = idesc_bf16(stacked ? 2 * n_query : n_query);
            const uint64_t a_desc0 = sdesc(saddr(kring)), b_desc0 = sdesc(saddr(qbuf));
            uint64_t a_step[8], b_step[8];
#pragma unroll
            for (int step = 0; step < 8; ++step) {
                const int half = step >> 2, kk = step & 3;
                a_step[step] = (uint64_t)((half * kHalfBytes + kk * 32) >> 4);
                b_step[step] = (uint64_t)((half * 2 * q_block + kk * 32) >> 4);
            }
            const uint64_t lo_step = q_block >> 4;
            uint32_t seq = 0, tcount = 0, qseq = 0;
            int64_t cur = -1;
            for (int64_t tile = walk.first; tile < walk.last; ++tile) {
                const int64_t head = tile / walk.tph;
                const int t0 = (int)(tile - head * walk.tph) * kTok;
                if (t0 >= head_len(seq_lens, head, heads, t_max, status, false)) continue;
                const uint32_t b = tcount & 1u, use = tcount >> 1;
                if (use > 0 && !bar_wait(&tempty[b], (use - 1) & 1u, status, &abort_flag, true)) break;
                fence_after();
                if (head != cur) {
                    if (qseq > 0) mma_commit(&qempty);  // the previous head's operand rows are free once its MMAs end
                    if (!bar_wait(&qfull, qseq & 1u, status, &abort_flag, true)) break;
                    ++qseq;
                    cur = head;
                }
                const int s = (int)(seq % (uint32_t)stages);
                if (!bar_wait(&full[s], (seq / stages) & 1u, status, &abort_flag, true)) break;
                fence_after();
                const uint32_t d_tmem = tmem + b * (uint32_t)acc_cols;
                const uint64_t a0 = a_desc0 + (uint64_t)((s * kTileBytes) >> 4);
                if (stacked) {
                    // one MMA per K-step: N = 2M operand rows (hi then lo)
#pragma unroll
                    for (int step = 0; step < 8; ++step)
                        mma_bf16(d_tmem, a0 + a_step[step], b_desc0 + b_step[step], idesc, step ? 1u : 0u);
                } else {
#pragma unroll
                    for (int step = 0; step < 8; ++step) {
                        mma_bf16(d_tmem, a0 + a_step[step], b_desc0 + b_step[step], idesc, step ? 1u : 0u);
                        mma_bf16(d_tmem, a0 + a_step[step], b_desc0 + b_step[step] + lo_step, idesc, 1u);
                    }
                }
                mma_commit(&empty[s]);
                mma_commit(&tfull[b]);
                ++seq;
                ++tcount;
            }
            // all MMAs issued by this thread complete before TMEM is freed
            mma_commit(&drain);
            bar_wait(&drain, 0, status, &abort_flag, false);
        }
    } else {
        // ----------------------------------------------------- epilogue --
        // Group g (warps 2-5: g = 0, warps 6-9: g = 1) sums query columns
        // [g * cw, (g + 1) * cw); group 1 hands its partial sums to group 0
        // through `part` (pready), and group 0 frees the accumulator buffer
        // only after reading them, so a slot of `part` is never rewritten
        // before it is read.
        const int grp = (warp - 2) >> 2;
        const uint32_t rank = (uint32_t)(warp & 3);  // TMEM lanes 32*rank .. 32*rank+31
        const int cw = n_query / groups;
        uint32_t tcount = 0;
        if (grp < groups) {
            for (int64_t tile = walk.first; tile < walk.last; ++tile) {
                const int64_t head = tile / walk.tph;
                const int t0 = (int)(tile - head * walk.tph) * kTok;
                const int T = head_len(seq_lens, head, heads, t_max, status, false);
                if (t0 >= T) continue;
                const uint32_t b = tcount & 1u, use = tcount >> 1;
                if (!bar_wait(&tfull[b], use & 1u, status, &abort_flag, true)) break;
                fence_after();
                const uint32_t taddr = tmem + ((rank * 32u) << 16) + b * (uint32_t)acc_cols;
                float acc = tmem_abs_sum(taddr, (uint32_t)n_query, stacked, grp * cw, cw);
                const int row = (int)rank * 32 + lane;
                if (grp == 1) {
                    part[b][row] = acc;
                    fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        bar_arrive(&pready[b]);
                        bar_arrive(&tempty[b]);
                    }
                } else {
                    if (groups == 2) {
                        if (!bar_wait(&pready[b], use & 1u, status, &abort_flag, true)) break;
                        acc += part[b][row];
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) bar_arrive(&tempty[b]);
                    const int t = t0 + row;
                    if (t < T) S[(size_t)head * t_max + t] = acc * scale;
                }
                ++tcount;
            }
        }
    }
    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
    }
}

// ------------------------------- 2b: the contraction on pairs of CTAs --
//
// k_oja_scores_pair: the same contraction with tcgen05.mma.cta_group::2 on a
// cluster of two CTAs, one per SM. One MMA covers 256 tokens: the CTA of
// cluster rank r holds tokens [128 r, 128 r + 128) of the tile (operand A)
// and operand split r (r = 0 the hi rows, r = 1 the lo rows: operand B, N =
// 2M) in its shared memory, and receives its 128 tokens x 2M accumulator
// columns in its own TMEM -- the one-CTA kernel's layout, so the epilogue
// is the same. Rank 0's MMA thread issues every MMA of the pair: for the
// same work each SM issues half as many MMAs, and each reads only its half
// of the operand rows.
//  * Each CTA's producer loads its own halves with TMA onto its own
//    barriers. In rank 1 a relay thread waits for each of those copies in
//    order and arrives on rank 0's peer_full / peer_qfull, so the MMA thread
//    sees both halves land, and each CTA can still wait out its own copies.
//  * The MMA thread commits a stage's, an operand's and an accumulator's
//    completion to the barriers of both CTAs at once (multicast commit).
//  * Both CTAs' epilogue warps release an accumulator buffer on rank 0's
//    tempty (rank 1's with remote arrives).
//  * Both CTAs allocate and free the TMEM together (cta_group::2); the pair
//    checks that both received the same address before any MMA.
// Every wait is bounded as in the one-CTA kernel; the pair meets at a
// cluster barrier after the setup and again before the TMEM is freed.
__device__ __forceinline__ uint32_t pair_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t pair_map(const void *p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void pair_arrive_remote(uint32_t caddr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

__device__ __forceinline__ uint32_t pair_ld_u32(uint32_t caddr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
    return v;
}

__device__ __forceinline__ void pair_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}

// Completion of the MMAs issued so far arrives on the barrier at the same
// offset in both CTAs of the pair.
__device__ __forceinline__ void mma_commit_pair(uint64_t *b)
{
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            saddr(b)),
        "h"(mask)
        : "memory");
}

// ... on this CTA's barrier only.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t *b)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(b))
                 : "memory");
}

// Instruction descriptor of kind::f16 for the pair: M = 256 (128 tokens per
// CTA), N = n.
__host__ __device__ constexpr uint32_t idesc_bf16_pair(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

constexpr int kPairTok = 2 * kTok;  // tokens of one pair MMA

__global__ void __launch_bounds__(kOjaThreads, 1)
k_oja_scores_pair(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                  const int32_t *__restrict__ seq_lens, int heads, int t_max, int64_t n_heads, int n_query, int stages,
                  uint32_t tmem_cols, float scale, float *__restrict__ S, uint32_t *status)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *kring = smem;                               // stages x 32 KB: this CTA's 128 tokens of each tile
    uint8_t *qbuf = smem + (size_t)stages * kTileBytes;  // [dims 0-63, 64-127][n_query rows x 128 B]: this CTA's split (room for both)
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], peer_full[kMaxStages], qfull, qempty,
        peer_qfull, tfull[2], tempty[2], pready[2], drain;
    __shared__ float part[2][kTok];
    __shared__ uint32_t tmem_base_sh, s_ok;
    __shared__ volatile uint32_t abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = pair_rank();
    const uint32_t q_block = (uint32_t)n_query * 128u;  // bytes of one dims half of this CTA's operand rows
    const int acc_cols = 2 * n_query;                    // hi then lo columns
    const int groups = n_query % 64 == 0 ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            bar_init(&full[s], 1);
            bar_init(&empty[s], 1);
            bar_init(&peer_full[s], 1);
        }
        bar_init(&qfull, 1);
        bar_init(&qempty, 1);
        bar_init(&peer_qfull, 1);
        for (int b = 0; b < 2; ++b) {
            bar_init(&tfull[b], 1);
            bar_init(&tempty[b], 2 * 4 * groups);
            bar_init(&pready[b], 4);
        }
        bar_init(&drain, 1);
        abort_flag = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base_sh)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    pair_sync();  // both CTAs' barriers and TMEM are set up
    fence_after();
    if (threadIdx.x == 0) {
        // the MMAs write both CTAs' accumulators at rank 0's address
        const uint32_t other = pair_ld_u32(pair_map(&tmem_base_sh, rank ^ 1u));
        s_ok = other == tmem_base_sh ? 1u : 0u;
        if (!s_ok && rank == 0) atomicOr(status, MKV_DEV_INTERNAL);
    }
    __syncthreads();
    const bool ok = s_ok != 0u;  // the same in both CTAs (a symmetric comparison)
    const uint32_t tmem = tmem_base_sh;
    // the pair's tiles of 256 tokens
    const int tph = (t_max + kPairTok - 1) / kPairTok;
    const int64_t total = n_heads * tph;
    const int64_t npairs = gridDim.x / 2, pair = blockIdx.x / 2;
    const int64_t first = total * pair / npairs, last = total * (pair + 1) / npairs;

    if (ok && warp == 0) {
        if (lane == 0) {
            // ------------------------------ TMA producer (this CTA's halves) --
            uint32_t seq = 0, qseq = 0;
            uint32_t last_parity[kMaxStages];
            int64_t cur = -1;
            for (int64_t tile = first; tile < last; ++tile) {
                const int64_t head = tile / tph;
                const int t0 = (int)(tile - head * tph) * kPairTok;
                if (t0 >= head_len(seq_lens, head, heads, t_max, status, false)) continue;
                if (head != cur) {
                    if (qseq > 0 && !bar_wait(&qempty, (qseq - 1) & 1u, status, &abort_flag, true)) break;
                    bar_expect(&qfull, 2u * q_block);
                    for (int half = 0; half < 2; ++half)
                        tma_load_2d(qbuf + half * q_block, &tmap_q, half * 64, (int)((head * 2 + rank) * n_query),
                                    &qfull);
                    ++qseq;
                    cur = head;
                }
                const int s = (int)(seq % (uint32_t)stages);
                if (seq >= (uint32_t)stages &&
                    !bar_wait(&empty[s], ((seq / stages) - 1) & 1u, status, &abort_flag, true))
                    break;
                bar_expect(&full[s], (uint32_t)kTileBytes);
                const int row = (int)(head * t_max + t0 + (int)rank * kTok);
                tma_load_2d(kring + (size_t)s * kTileBytes, &tmap_k, 0, row, &full[s]);
                tma_load_2d(kring + (size_t)s * kTileBytes + kHalfBytes, &tmap_k, 64, row, &full[s]);
                last_parity[s] = (seq / stages) & 1u;
                ++seq;
            }
            // every copy issued lands before the CTA may exit
            const uint32_t issued = seq < (uint32_t)stages ? seq : (uint32_t)stages;
            for (uint32_t s = 0; s < issued; ++s) bar_wait(&full[s], last_parity[s], status, &abort_flag, false);
            if (qseq > 0) bar_wait(&qfull, (qseq - 1) & 1u, status, &abort_flag, false);
        }
    } else if (ok && warp == 1) {
        if (lane == 0 && rank == 1) {
            // ----------------------------------- relay (rank 1): copies landed --
            const uint32_t pf0 = pair_map(&peer_full[0], 0), pq = pair_map(&peer_qfull, 0);
            uint32_t seq = 0, qseq = 0;
            int64_t cur = -1;
            for (int64_t tile = first; tile < last; ++tile) {
                const int64_t head = tile / tph;
                const int t0 = (int)(tile - head * tph) * kPairTok;
                if (t0 >= head_len(seq_lens, head, heads, t_max, status, false)) continue;
                if (head != cur) {
                    if (!bar_wait(&qfull, qseq & 1u, status, &abort_flag, true)) break;
                    pair_arrive_remote(pq);
                    ++qseq;
                    cur = head;
                }
                const int s = (int)(seq % (uint32_t)stages);
                if (!bar_wait(&full[s], (seq / stages) & 1u, status, &abort_flag, true)) break;
                pair_arrive_remote(pf0 + (uint32_t)(s * sizeof(uint64_t)));
                ++seq;
            }
        } else if (lane == 0 && rank == 0) {
            // ---------------------------------------------- MMA issuer (pair) --
            const uint32_t idesc = idesc_bf16_pair(2 * n_query);
            const uint64_t a_desc0 = sdesc(saddr(kring)), b_desc0 = sdesc(saddr(qbuf));
            uint64_t a_step[8], b_step[8];
#pragma unroll
            for (int step = 0; step < 8; ++step) {
                const int half = step >> 2, kk = step & 3;
                a_step[step] = (uint64_t)((half * kHalfBytes + kk * 32) >> 4);
                b_step[step] = (uint64_t)((half * q_block + kk * 32) >> 4);
            }
            uint32_t seq = 0, tcount = 0, qseq = 0;
            int64_t cur = -1;
            for (int64_t tile = first; tile < last; ++tile) {
                const int64_t head = tile / tph;
                const int t0 = (int)(tile - head * tph) * kPairTok;
                if (t0 >= head_len(seq_lens, head, heads, t_max, status, false)) continue;
                const uint32_t b = tcount & 1u, use = tcount >> 1;
                if (use > 0 && !bar_wait(&tempty[b], (use - 1) & 1u, status, &abort_flag, true)) break;
                fence_after();
                if (head != cur) {
                    if (qseq > 0) mma_commit_pair(&qempty);  // the previous head's operand rows are free in both CTAs
                    if (!bar_wait(&qfull, qseq & 1u, status, &abort_flag, true) ||
                        !bar_wait(&peer_qfull, qseq & 1u, status, &abort_flag, true))
                        break;
                    ++qseq;
                    cur = head;
                }
                const int s = (int)(seq % (uint32_t)stages);
                if (!bar_wait(&full[s], (seq / stages) & 1u, status, &abort_flag, true) ||
                    !bar_wait(&peer_full[s], (seq / stages) & 1u, status, &abort_flag, true))
                    break;
                fence_after();
                const uint32_t d_tmem = tmem + b * (uint32_t)acc_cols;
                const uint64_t a0 = a_desc0 + (uint64_t)((s * kTileBytes) >> 4);
#pragma unroll
                for (int step = 0; step < 8; ++step)
                    mma_bf16_pair(d_tmem, a0 + a_step[step], b_desc0 + b_step[step], idesc, step ? 1u : 0u);
                mma_commit_pair(&empty[s]);
                mma_commit_pair(&tfull[b]);
                ++seq;
                ++tcount;
            }
            // every MMA issued completes before the TMEM is freed
            mma_commit_pair_local(&drain);
            bar_wait(&drain, 0, status, &abort_flag, false);
        }
    } else if (ok) {
        // ----------------------------------------------------- epilogue --
        // as in the one-CTA kernel; rank 1's warps release a buffer on rank
        // 0's tempty
        const int grp = (warp - 2) >> 2;
        const uint32_t wq = (uint32_t)(warp & 3);  // TMEM lanes 32*wq .. 32*wq+31
        const int cw = n_query / groups;
        const uint32_t te0 = pair_map(&tempty[0], 0);
        auto release = [&](uint32_t b) {
            if (rank == 0)
                bar_arrive(&tempty[b]);
            else
                pair_arrive_remote(te0 + b * (uint32_t)sizeof(uint64_t));
        };
        uint32_t tcount = 0;
        if (grp < groups) {
            for (int64_t tile = first; tile < last; ++tile) {
                const int64_t head = tile / tph;
                const int t0 = (int)(tile - head * tph) * kPairTok;
                const int T = head_len(seq_lens, head, heads, t_max, status, false);
                if (t0 >= T) continue;
                const uint32_t b = tcount & 1u, use = tcount >> 1;
                if (!bar_wait(&tfull[b], use & 1u, status, &abort_flag, true)) break;
                fence_after();
                const uint32_t taddr = tmem + ((wq * 32u) << 16) + b * (uint32_t)acc_cols;
                float acc = tmem_abs_sum(taddr, (uint32_t)n_query, true, grp * cw, cw);
                const int row = (int)wq * 32 + lane;
                if (grp == 1) {
                    part[b][row] = acc;
                    fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        bar_arrive(&pready[b]);
                        release(b);
                    }
                } else {
                    if (groups == 2) {
                        if (!bar_wait(&pready[b], use & 1u, status, &abort_flag, true)) break;
                        acc += part[b][row];
                    }
                    fence_before();
                    __syncwarp();
                    if (lane == 0) release(b);
                    const int t = t0 + (int)rank * kTok + row;
                    if (t < T) S[(size_t)head * t_max + t] = acc * scale;
                }
                ++tcount;
            }
        }
    }
    fence_before();
    __syncthreads();
    pair_sync();  // every MMA and every TMEM read of both CTAs is done
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
    }
}

// --------------------------------------------------------------- host side --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, 128] with 256-byte rows; boxes of 64 dims x box_rows
// rows in the 128-byte swizzle layout.
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
    const cuuint32_t box[2] = {64u, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sms_of_current_device()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

size_t oja_operand_bytes(int64_t n_heads, int32_t n_query)
{
    return (size_t)n_heads * 2 * (size_t)n_query * kRowBytes;
}

// The CTA-pair contraction (k_oja_scores_pair) for n_query <= 128 (hi and
// lo stacked in one MMA): 0 never, 1 wherever it applies.
std::atomic<int> g_oja_pair{0};

int oja_set_pair(int enable) { return g_oja_pair.exchange(enable ? 1 : 0); }

bool oja_uses_pair(int32_t n_query) { return g_oja_pair.load(std::memory_order_relaxed) != 0 && 2 * n_query <= 256; }

// stages of the pair kernel: each CTA loads one split (hi or lo) of the
// operand rows; the operand buffer keeps the one-CTA kernel's size (both
// splits), so the MMA's operand reads stay inside the CTA's shared memory
// whatever rows it addresses
int oja_pair_stages(int32_t n_query)
{
    const int left = kSmemBudget - 1024 - 2048 - 4 * n_query * 128;
    const int s = left / kTileBytes;
    return s > kMaxStages ? kMaxStages : s;
}

int oja_stages(int32_t n_query)
{
    // alignment slack, up to 2 KB of static shared memory, the operand rows
    const int left = kSmemBudget - 1024 - 2048 - 4 * n_query * 128;
    const int s = left / kTileBytes;
    return s > kMaxStages ? kMaxStages : s;
}

cudaError_t launch_oja_scores(const Geometry &g, const void *K, const void *Q, const float *U, const int32_t *seq_lens,
                              int32_t n_query, int32_t rank, void *qhl, float *S, uint32_t *status, cudaStream_t st,
                              void *const *events)
{
    if (g.n_heads == 0 || g.t_max == 0) return cudaSuccess;
    auto mark = [&](int i) -> cudaError_t {
        return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st) : cudaSuccess;
    };
    cudaError_t e;
    if ((e = mark(0)) != cudaSuccess) return e;
    // 1: projected query rows, hi + lo
    const int rows = n_query % 64 == 0 ? 64 : (n_query % 32 == 0 ? 32 : 16);
    const int64_t items = g.n_heads * (n_query / rows);
    const int pthreads = rows / kProjBlock * 32;
    const size_t psmem =
        (size_t)(rows * kProjQStride + kHeadDim * proj_u_stride(rank) + rows * proj_rank_pad(rank)) * sizeof(float);
    e = cudaFuncSetAttribute(k_oja_project, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return e;
    const int pgrid = grid_for_items(reinterpret_cast<const void *>(k_oja_project), pthreads, psmem, items);
    k_oja_project<<<pgrid, pthreads, psmem, st>>>(static_cast<const __nv_bfloat16 *>(Q), U, n_query, rank, rows,
                                                      items, static_cast<__nv_bfloat16 *>(qhl));
    if ((e = cudaGetLastError()) != cudaSuccess || (e = mark(1)) != cudaSuccess) return e;
    // 2: the contraction
    CUtensorMap mk, mq;
    if (!make_map(&mk, K, (uint64_t)g.n_heads * g.t_max, kTok) ||
        !make_map(&mq, qhl, (uint64_t)g.n_heads * 2 * n_query, (uint32_t)n_query))
        return cudaErrorInvalidValue;
    const float scale = (float)(1.0 / ((double)n_query * 11.313708498984760390));  // 1 / (M sqrt(128))
    const int sms = sms_of_current_device();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (oja_uses_pair(n_query)) {
        // pairs of CTAs (a cluster of two, one CTA per SM), 256 tokens per MMA
        const int pstages = oja_pair_stages(n_query);
        if (pstages < 2) return cudaErrorInvalidValue;
        const size_t psmem2 = 1024 + (size_t)pstages * kTileBytes + 4 * (size_t)n_query * 128;
        const void *fn = reinterpret_cast<const void *>(k_oja_scores_pair);
        if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem2)) != cudaSuccess)
            return e;
        uint32_t pcols = 32;
        while (pcols < (uint32_t)(2 * 2 * n_query)) pcols *= 2;  // two accumulator buffers of 2M columns
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kOjaThreads);
        cfg.dynamicSmemBytes = psmem2;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2);
        int max_pairs = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&max_pairs, fn, &cfg)) != cudaSuccess) return e;
        if (max_pairs < 1) return cudaErrorInvalidConfiguration;
        const int64_t ptiles = g.n_heads * ((g.t_max + 2 * kTok - 1) / (2 * kTok));
        const int pairs = (int)(ptiles < max_pairs ? ptiles : max_pairs);
        cfg.gridDim = dim3((unsigned)(2 * pairs));
        const int32_t *sl = seq_lens;
        int heads = g.heads, t_max = g.t_max, nq = n_query, stg = pstages;
        int64_t nh = g.n_heads;
        void *args[] = {&mk, &mq, &sl, &heads, &t_max, &nh, &nq, &stg, &pcols, const_cast<float *>(&scale), &S,
                        &status};
        if ((e = cudaLaunchKernelExC(&cfg, fn, args)) != cudaSuccess) return e;
        return mark(2);
    }
    const int stages = oja_stages(n_query);
    if (stages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)stages * kTileBytes + 4 * (size_t)n_query * 128;
    if ((e = cudaFuncSetAttribute(k_oja_scores, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    // independent accumulators per tile: as many (up to 4) as two buffers of
    // them fit in the 512 TMEM columns
    // two accumulator buffers of 2M columns (hi and lo side by side) for
    // M <= 128, of M columns (hi and lo summed by the MMAs) above
    const int acc_cols = 2 * n_query <= 256 ? 2 * n_query : n_query;
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * acc_cols)) cols *= 2;
    const int64_t tiles = g.n_heads * ((g.t_max + kTok - 1) / kTok);
    const int grid = (int)(tiles < sms ? tiles : sms);
    k_oja_scores<<<grid, kOjaThreads, smem, st>>>(mk, mq, seq_lens, g.heads, g.t_max, g.n_heads, n_query, stages, cols,
                                                  scale, S, status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return mark(2);
}

}  // namespace mkv
