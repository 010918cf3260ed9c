// Prefill dense contraction on a Q8_0 activation image (minfer doc 52, "r49
// A-quantize prepass shared-A dedup", sections 1 and 5: the q/k/v and
// gate/up GEMMs that read one quantised A).
//
//   C[t][n] = sum_b d_w[n][b] * d_a[t][b] * sum_{i in b} (nibble_i - 8) * q_i
//
// On the 5th-generation tensor cores (tcgen05.mma kind::f16, accumulator in
// tensor memory). Both operands enter as binary16 values of the dequantised
// blocks, each rounded once: A[n][k] = f16((nibble - 8) * d_w) and
// B[t][k] = f16(q * d_a), and the MMA accumulates over all of K in binary32.
// The pages scale an exact int8 block dot in f32 instead; the two agree to
// about 2^-11 relative per product (NMSE ~1e-7), far inside their 5e-4 bound.
// (tcgen05 kind::i8 does not exist on sm_103a, and applying the scales block
// by block from tensor memory would bound the kernel by FP32 issue.)
//
// Two kernels per call:
//   dequant_b: the image -> B, [T][K] binary16 in the caller's workspace,
//     once per call (it is read by every 128-row weight tile).
//   mmq_tc: persistent, one CTA per SM, tiles of (projection, 128-row weight
//     tile, 256-token tile) taken round-robin, tokens fastest so that the CTAs
//     running at one time share a few weight row tiles through L2.
//     A stage is one packed unit: 128 K elements, B as two 64-column boxes
//     (64 KB), A as 64 tensor-memory columns, eight MMAs; three stages.
//     (Stages of 64 K elements measured 6-11% slower: each stage pays a fixed
//     round of barrier hand-offs between the warps below.)
//     warp 0: TMA -- the B tiles (2D tensor copies, 128-byte swizzle) and the
//             packed weight units (bulk copies) into shared-memory rings, with
//             L2 prefetches of the units a few ahead;
//     warps 2-9: turn each unit's nibbles into f16 A stages held in tensor
//             memory (tcgen05.st; two warps per 32-lane quarter, two 32-blocks
//             each), so the MMAs read A from tensor memory and only B from
//             shared memory;
//     warp 1: allocates tensor memory (one 256-column accumulator and three
//             64-column A stages) and issues the MMAs (one thread);
//     warps 10-25: read the finished accumulator (64 columns of one lane
//             quarter per warp), release it to the next tile's MMAs before
//             storing anything, then store C (8 warps that stored their first
//             64 columns before reading the second held the next tile's MMAs
//             back by about 7% on the gate/up launch).
// Within a 32-block the K positions follow the order in which the converters
// store a packed weight word (column 2t+p: elements 4t+p and 4t+p+2; column
// 8+2t+p: elements 16+4t+p and 18+4t+p); dequant_b writes B in the same order.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "qk_internal.cuh"

namespace qk {
namespace {

constexpr int MAX_PROJ = 8;
constexpr int TM = 128;              // weight rows per CTA (MMA M)
constexpr int TN = 256;              // tokens per CTA (MMA N; 3325 tokens = 13 tiles)
constexpr int KC = 64;               // K elements of one B box (one 128-byte swizzle row of f16)
constexpr int SK = 128;              // K elements per stage: one packed unit, two B boxes
constexpr int NS = 3;                // stages (A in tensor memory, B in shared memory)
constexpr int NU = 3;                // packed-unit staging slots (a unit = one stage)
constexpr int PF = 10;               // units prefetched into L2 ahead of the one being loaded
constexpr int B_BOX = TN * KC * 2;   // 32 KB
constexpr int B_TILE = TN * SK * 2;  // 64 KB
constexpr uint32_t A_COLS = SK / 2;  // tensor-memory columns of one A stage (two f16 per column)
constexpr int EPI0 = 10;             // first epilogue warp
constexpr int N_EPI = 16;            // epilogue warps: 4 lane quarters x 4 column quarters of 64
constexpr int THREADS = (EPI0 + N_EPI) * 32;
constexpr uint32_t A_TMEM = TN;           // A stages follow the accumulator
constexpr uint32_t TMEM_COLS = 512;
static_assert(A_TMEM + NS * A_COLS <= TMEM_COLS, "tensor memory");
constexpr uint32_t SPIN_LIMIT = 1u << 16;
constexpr uint32_t SUSPEND_NS = 20000;

// shared memory: [B tiles][units][barriers][tensor-memory address]
constexpr int OFF_B = 0;
constexpr int OFF_U = OFF_B + NS * B_TILE;
constexpr int OFF_BAR = OFF_U + NU * Q4_UNIT_BYTES;
// full_a[NS] full_b[NS] empty[NS] ufull[NU] uempty[NU] acc_full acc_empty mma_done
constexpr int N_BARS = 3 * NS + 2 * NU + 3;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + slack to align the base to 1024
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// instruction descriptor: f32 accumulator, f16 A and B, both K-major, N = 256, M = 128
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);

__device__ unsigned int g_mmq_faults = 0;

struct MmqProj {
    const uint8_t *w;
    float *y;
    int64_t y_stride;
    int N, K, chunks, row_tiles, rt_begin;   // rt_begin: first global row tile
};
struct MmqArgs {
    CUtensorMap bmap;    // B [T][K] f16, box 64 x 256, 128-byte swizzle
    int T, n_proj, tok_tiles, tiles;
    MmqProj p[MAX_PROJ];
};
struct Tile {
    int j, rt, tok0, nkc;
};
__device__ __forceinline__ Tile tile_of(const MmqArgs &a, int tau) {
    Tile t;
    const int r = tau / a.tok_tiles;
    t.tok0 = (tau - r * a.tok_tiles) * TN;
    int j = 0;
    while (j + 1 < a.n_proj && r >= a.p[j + 1].rt_begin) j++;
    t.j = j;
    t.rt = r - a.p[j].rt_begin;
    t.nkc = (a.p[j].K + SK - 1) / SK;   // stages = packed units
    return t;
}

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
// Bounded wait: suspends until the phase completes (or SUSPEND_NS), gives up
// after SPIN_LIMIT tries (about a second at most), records a fault and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
    for (uint32_t i = 0; i < SPIN_LIMIT; i++) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity), "r"(SUSPEND_NS)
            : "memory");
        if (ok) return true;
    }
    atomicOr(&g_mmq_faults, 1u);
    return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
        : "memory");
}
// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
// D (tensor memory) (+)= A (tensor memory) x B (shared memory)
__device__ __forceinline__ void tc_mma(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tmem),
        "r"(a_tmem), "l"(b), "r"(IDESC), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Four weight bytes (word t of one row of a Q4_0 block) -> 16 bytes of f16
// A values (nibble - 8) * dw, K order: e(4t), e(4t+2), e(4t+1), e(4t+3),
// e(16+4t), e(16+4t+2), e(16+4t+1), e(16+4t+3). The nibble becomes an exact
// half by OR-ing it under an exponent (1024 + lo, 64 + hi); subtracting
// 1032 / 72 leaves the exact nibble - 8; one rounding in the multiply by dw.
__device__ __forceinline__ uint32_t a_pair(uint32_t v, __half2 bias, __half2 dw) {
    const __half2 r = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&v), bias), dw);
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint4 a_word(uint32_t w, __half2 dw) {
    const uint32_t w8 = w >> 8;
    const __half2 blo = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    const __half2 bhi = __halves2half2(__ushort_as_half(0x5480), __ushort_as_half(0x5480));   // 72
    return make_uint4(a_pair((w & 0x000F000Fu) | 0x64006400u, blo, dw), a_pair((w8 & 0x000F000Fu) | 0x64006400u, blo, dw),
                      a_pair((w & 0x00F000F0u) | 0x54005400u, bhi, dw),
                      a_pair((w8 & 0x00F000F0u) | 0x54005400u, bhi, dw));
}

// ------------------------------------------------------------------ B = dequantised image
// Two codes of word v (bytes k and k + 2, k = 0 or 1) -> f16 pair q * d_a. A code becomes an
// exact half by placing its biased byte (q + 128) under the exponent of 1024 (PRMT); subtracting
// 1152 leaves q exactly; the binary16 multiply by d_a rounds the exact product once, as the
// binary32 product rounded to binary16 would.
__device__ __forceinline__ uint32_t b_pair(uint32_t u, uint32_t sel, __half2 d2) {
    uint32_t h;
    asm("prmt.b32 %0, %1, 0x64646464, %2;" : "=r"(h) : "r"(u), "r"(sel));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    const __half2 r = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&h), bias), d2);
    return *reinterpret_cast<const uint32_t *>(&r);
}
// four codes (one word, elements e .. e+3) -> halves in the order e, e+2, e+1, e+3
__device__ __forceinline__ uint2 b_word(uint32_t v, __half2 d2) {
    const uint32_t u = v ^ 0x80808080u;   // q + 128 in each byte
    return make_uint2(b_pair(u, 0x4240u, d2), b_pair(u, 0x4341u, d2));
}

// grid (T, ceil(4 kb / 256)), tokens on x: thread j of CTA (t, y) takes word w = j & 3 of block
// b = 64 y + j / 4 of token t: codes 4w .. 4w+3 and 16+4w .. 16+4w+3 -> f16 q * d_a at columns
// 2w, 2w+1 (halves 4w .. 4w+3) and 8+2w, 9+2w (halves 16+4w ..), the K order of the A stages.
__global__ void __launch_bounds__(256) dequant_b_kernel(const int8_t *__restrict__ qs, const uint16_t *__restrict__ d,
                                                        int64_t row_blocks, int T, int kb, __half *__restrict__ B) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x, w = threadIdx.x & 3, b = blockIdx.y * 64 + (threadIdx.x >> 2);
    if (b >= kb) return;
    const int8_t *src = qs + ((int64_t)t * row_blocks + b) * QB;
    const uint32_t lo = __ldg(reinterpret_cast<const unsigned int *>(src + 4 * w));
    const uint32_t hi = __ldg(reinterpret_cast<const unsigned int *>(src + 16 + 4 * w));
    const __half dah = __ushort_as_half(__ldg(d + (int64_t)t * row_blocks + b));
    const __half2 d2 = __halves2half2(dah, dah);
    __half *dst = B + ((int64_t)t * kb + b) * QB;
    *reinterpret_cast<uint2 *>(dst + 4 * w) = b_word(lo, d2);
    *reinterpret_cast<uint2 *>(dst + 16 + 4 * w) = b_word(hi, d2);
}

// ------------------------------------------------------------------ the GEMM
__global__ void __launch_bounds__(THREADS, 1) mmq_tc_kernel(const __grid_constant__ MmqArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_a = sbase + OFF_BAR, full_b = full_a + NS * 8, empty = full_b + NS * 8;
    const uint32_t ufull = empty + NS * 8, uempty = ufull + NU * 8, acc_full = uempty + NU * 8,
                   acc_empty = acc_full + 8, mma_done = acc_empty + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + N_BARS * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(full_a + 8 * s, 256);   // the eight converter warps
            mbar_init(full_b + 8 * s, 1);     // the producer, with the bytes
            mbar_init(empty + 8 * s, 1);      // the MMA commit
        }
        for (int u = 0; u < NU; u++) {
            mbar_init(ufull + 8 * u, 1);
            mbar_init(uempty + 8 * u, 256);
        }
        mbar_init(acc_full, 1);      // the MMA commit after a tile's last stage
        mbar_init(acc_empty, N_EPI * 32);   // the epilogue warps, once they have read it
        mbar_init(mma_done, 1);      // the MMA thread's last commit: all its MMAs are done
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {   // tensor memory: the accumulator (256 columns) and A stages (3 x 64 columns)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();
    pdl_wait();   // B comes from the previous kernel

    if (warp == 0) {   // ---------------- producer
        if (lane == 0) {
            uint32_t g = 0, gu = 0;   // stages and units issued by this CTA
            bool ok = true;
            {   // L2 prefetch of the first tile's leading units
                const Tile t = tile_of(a, blockIdx.x < a.tiles ? blockIdx.x : 0);
                const MmqProj &P = a.p[t.j];
                const uint8_t *units = P.w + (int64_t)t.rt * P.chunks * Q4_UNIT_BYTES;
                for (int u = 0; u < PF && u < P.chunks && (int)blockIdx.x < a.tiles; u++)
                    prefetch_l2(units + (int64_t)u * Q4_UNIT_BYTES, Q4_UNIT_BYTES);
            }
            for (int tau = blockIdx.x; tau < a.tiles && ok; tau += G) {
                const Tile t = tile_of(a, tau);
                const MmqProj &P = a.p[t.j];
                const uint8_t *units = P.w + (int64_t)t.rt * P.chunks * Q4_UNIT_BYTES;
                for (int kc = 0; kc < t.nkc; kc++, g++) {   // stage kc = packed unit kc
                    const uint32_t s = g % NS;
                    {
                        const int u = kc;
                        const uint32_t us = gu % NU;
                        if (gu >= NU && !mbar_wait(uempty + 8 * us, ((gu / NU) - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(ufull + 8 * us, Q4_UNIT_BYTES);
                        bulk_g2s(sbase + OFF_U + us * Q4_UNIT_BYTES, units + (int64_t)u * Q4_UNIT_BYTES,
                                 Q4_UNIT_BYTES, ufull + 8 * us);
                        gu++;
                        // keep the unit PF ahead (in this tile or the next one) on its way into L2
                        if (u + PF < P.chunks) {
                            prefetch_l2(units + (int64_t)(u + PF) * Q4_UNIT_BYTES, Q4_UNIT_BYTES);
                        } else if (tau + G < a.tiles) {
                            const Tile n = tile_of(a, tau + G);
                            const MmqProj &Q = a.p[n.j];
                            const int un = u + PF - P.chunks;
                            if (un < Q.chunks)
                                prefetch_l2(Q.w + ((int64_t)n.rt * Q.chunks + un) * Q4_UNIT_BYTES, Q4_UNIT_BYTES);
                        }
                    }
                    if (g >= NS && !mbar_wait(empty + 8 * s, ((g / NS) - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    // the stage's B: two 64-column boxes (past K they read as zeros)
                    mbar_expect_tx(full_b + 8 * s, B_TILE);
                    tma_2d(sbase + OFF_B + s * B_TILE, &a.bmap, kc * SK, t.tok0, full_b + 8 * s);
                    tma_2d(sbase + OFF_B + s * B_TILE + B_BOX, &a.bmap, kc * SK + KC, t.tok0, full_b + 8 * s);
                }
            }
            // Every copy this thread issued has landed before the CTA can exit, also after a wait
            // above ran out: the last NS stages' B and the last NU units (a barrier whose phase
            // completed long ago passes at once). A wait that runs out here ends the drain.
            for (uint32_t x = g > NS ? g - NS : 0; x < g; x++)
                if (!mbar_wait(full_b + 8 * (x % NS), (x / NS) & 1u)) break;
            for (uint32_t x = gu > NU ? gu - NU : 0; x < gu; x++)
                if (!mbar_wait(ufull + 8 * (x % NU), (x / NU) & 1u)) break;
        }
    } else if (warp == 1) {   // ---------------- MMA issue (one thread)
        if (lane == 0) {
            uint32_t g = 0;
            int i = 0;
            bool ok = true;
            for (int tau = blockIdx.x; tau < a.tiles && ok; tau += G, i++) {
                const Tile t = tile_of(a, tau);
                const uint32_t acc = tmem;
                if (i >= 1 && !mbar_wait(acc_empty, (i - 1) & 1u)) break;
                tc_fence_after();
                for (int kc = 0; kc < t.nkc; kc++, g++) {
                    const uint32_t s = g % NS, par = (g / NS) & 1u;
                    if (!mbar_wait(full_a + 8 * s, par) || !mbar_wait(full_b + 8 * s, par)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t at = tmem + A_TMEM + s * A_COLS, bt = sbase + OFF_B + s * B_TILE;
#pragma unroll
                    for (int ks = 0; ks < SK / 16; ks++)   // K = 16 per MMA: 8 A columns, 32 B bytes of a box
                        tc_mma(acc, at + 8 * ks, sdesc(bt + (ks >> 2) * B_BOX + 32 * (ks & 3)), (kc | ks) != 0);
                    tc_commit(empty + 8 * s);   // frees the stage once these MMAs are done
                }
                if (ok) tc_commit(acc_full);   // the accumulator is final once its MMAs are done
            }
            // every MMA issued here is complete before the tensor memory is freed (after a wait
            // that ran out as well)
            tc_commit(mma_done);
            mbar_wait(mma_done, 0u);
        }
    } else if (warp < EPI0) {   // ---------------- warps 2..9: A conversion into tensor memory
        // A warp may only touch tensor-memory lanes 32 (warp % 4) .. +31: its rows are tile rows
        // 32 (warp % 4) .. +31, region warp % 4 of the packed unit, and tensor-memory lane = tile row.
        const int quad = warp & 3, qb = (warp - 2) >> 2;   // qb: the stage's block this warp converts
        const uint32_t arow = tmem + ((uint32_t)(32 * quad) << 16) + A_TMEM;
        uint32_t g = 0, gu = 0;
        bool ok = true;
        for (int tau = blockIdx.x; tau < a.tiles && ok; tau += G) {
            const Tile t = tile_of(a, tau);
            for (int kc = 0; kc < t.nkc; kc++, g++) {   // stage kc = packed unit kc
                const uint32_t s = g % NS, us = gu % NU;
                ok = mbar_wait(ufull + 8 * us, (gu / NU) & 1u);
                if (ok && g >= NS) ok = mbar_wait(empty + 8 * s, ((g / NS) - 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint8_t *unit = smem + OFF_U + us * Q4_UNIT_BYTES;
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    // Lane (g, t) loads word t of rows g, g+8, 16+g, 24+g of the warp's 32 rows (one
                    // conflict-free 16-byte load) and stores them with the 16x256b shape: registers 0,1
                    // go to lane g and 2,3 to lane g+8 at columns 2t, 2t+1, registers 4..7 the same way
                    // at columns 8+2t, 9+2t; a second store does lanes 16+g and 24+g. So column 2t+p of a
                    // block holds elements (4t+p, 4t+p+2) and column 8+2t+p holds (16+4t+p, 18+4t+p).
                    const int jb = 2 * h + qb, gq = lane >> 2;
                    const uint4 wv = *reinterpret_cast<const uint4 *>(unit + jb * 2048 + quad * 512 + lane * 16);
                    const uint2 sc = *reinterpret_cast<const uint2 *>(unit + 8192 + jb * 256 + gq * 32 + quad * 8);
                    const __half2 s01 = *reinterpret_cast<const __half2 *>(&sc.x), s23 = *reinterpret_cast<const __half2 *>(&sc.y);
                    const uint4 a0 = a_word(wv.x, __low2half2(s01)), a1 = a_word(wv.y, __high2half2(s01));
                    const uint4 a2 = a_word(wv.z, __low2half2(s23)), a3 = a_word(wv.w, __high2half2(s23));
                    const uint32_t base = arow + s * A_COLS + 16 * jb;
                    asm volatile(
                        "tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(base),
                        "r"(a0.x), "r"(a0.y), "r"(a1.x), "r"(a1.y), "r"(a0.z), "r"(a0.w), "r"(a1.z), "r"(a1.w)
                        : "memory");
                    asm volatile(
                        "tcgen05.st.sync.aligned.16x256b.x2.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(base + (16u << 16)),
                        "r"(a2.x), "r"(a2.y), "r"(a3.x), "r"(a3.y), "r"(a2.z), "r"(a2.w), "r"(a3.z), "r"(a3.w)
                        : "memory");
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                mbar_arrive(full_a + 8 * s);
                mbar_arrive(uempty + 8 * us);
                gu++;
            }
        }
    } else {   // ---------------- warps 10..25: epilogue (accumulator lane = tile row, column = token)
        // warp w reads lanes 32 (w % 4).. of columns 64 ((w - 10) / 4) ..+63 in one load and releases
        // the accumulator before storing anything, so the next tile's MMAs start while C is written
        const int quad = warp & 3, c0 = ((warp - EPI0) >> 2) * 64;
        int i = 0;
        for (int tau = blockIdx.x; tau < a.tiles; tau += G, i++) {
            const Tile t = tile_of(a, tau);
            const MmqProj &P = a.p[t.j];
            if (!mbar_wait(acc_full, i & 1u)) break;
            tc_fence_after();
            const int row = t.rt * TM + quad * 32 + lane;
            uint32_t v[64];
            const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0;
#pragma unroll
            for (int h = 0; h < 2; h++)   // two 32-column loads (a 64-column load needs more registers)
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                    "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                    : "=r"(v[32 * h + 0]), "=r"(v[32 * h + 1]), "=r"(v[32 * h + 2]), "=r"(v[32 * h + 3]),
                      "=r"(v[32 * h + 4]), "=r"(v[32 * h + 5]), "=r"(v[32 * h + 6]), "=r"(v[32 * h + 7]),
                      "=r"(v[32 * h + 8]), "=r"(v[32 * h + 9]), "=r"(v[32 * h + 10]), "=r"(v[32 * h + 11]),
                      "=r"(v[32 * h + 12]), "=r"(v[32 * h + 13]), "=r"(v[32 * h + 14]), "=r"(v[32 * h + 15]),
                      "=r"(v[32 * h + 16]), "=r"(v[32 * h + 17]), "=r"(v[32 * h + 18]), "=r"(v[32 * h + 19]),
                      "=r"(v[32 * h + 20]), "=r"(v[32 * h + 21]), "=r"(v[32 * h + 22]), "=r"(v[32 * h + 23]),
                      "=r"(v[32 * h + 24]), "=r"(v[32 * h + 25]), "=r"(v[32 * h + 26]), "=r"(v[32 * h + 27]),
                      "=r"(v[32 * h + 28]), "=r"(v[32 * h + 29]), "=r"(v[32 * h + 30]), "=r"(v[32 * h + 31])
                    : "r"(taddr + 32u * h));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(acc_empty);   // read: the MMAs of the next tile may start
            const int ntok = a.T - (t.tok0 + c0);   // tokens of this column quarter that exist
            if (row < P.N && ntok > 0) {
                float *yp = P.y + (int64_t)(t.tok0 + c0) * P.y_stride + row;
                const int64_t step = P.y_stride;
#pragma unroll
                for (int k = 0; k < 64; k++, yp += step)
                    if (k < ntok) *yp = __uint_as_float(v[k]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                     : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

int64_t mmq_workspace_bytes(int64_t T, int64_t kmax) { return (T * kmax * 2 + 127) / 128 * 128; }

qk_status read_mmq_faults(uint32_t *faults) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_mmq_faults, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_mmq_faults, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "qk_device_faults: %s", cudaGetErrorString(e));
    *faults = v;
    return QK_OK;
}

qk_status launch_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int T, int n_proj,
                     const qk_proj *projs, void *ws, size_t ws_bytes, cudaStream_t s) {
    MmqArgs a = {};
    a.T = T;
    a.n_proj = n_proj;
    int rtiles = 0, kmax = 0;
    for (int j = 0; j < n_proj; j++) {
        MmqProj &p = a.p[j];
        p.w = static_cast<const uint8_t *>(projs[j].w);
        p.y = projs[j].y;
        p.y_stride = projs[j].y_stride;
        p.N = (int)projs[j].N;
        p.K = (int)projs[j].K;
        p.chunks = (int)ceil_div(p.K, UNIT_COLS);
        p.row_tiles = (int)ceil_div(p.N, UNIT_ROWS);
        p.rt_begin = rtiles;
        rtiles += p.row_tiles;
        kmax = p.K > kmax ? p.K : kmax;
    }
    if (!ws || ws_bytes < (size_t)mmq_workspace_bytes(T, kmax))
        return fail(QK_ERR_WORKSPACE, "mmq: workspace %zu < %lld bytes", ws_bytes,
                    (long long)mmq_workspace_bytes(T, kmax));
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(QK_ERR_CUDA, "mmq: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)kmax, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)kmax * 2};
    const cuuint32_t box[2] = {KC, TN}, estr[2] = {1, 1};
    const CUresult r = enc(&a.bmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, ws, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QK_ERR_CUDA, "mmq: tensor map encoding failed (%d)", (int)r);

    const int kb = kmax / QB;
    qk_status st = launch_pdl("mmq_dequant_b", dequant_b_kernel, dim3((unsigned)T, (unsigned)ceil_div(kb, 64)),
                              dim3(256), 0, s, qs, d, row_blocks, T, kb, static_cast<__half *>(ws));
    if (st != QK_OK) return st;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(mmq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return fail(QK_ERR_CUDA, "mmq: shared memory attribute: %s", cudaGetErrorString(e));
        configured = true;
    }
    a.tok_tiles = (int)ceil_div(T, TN);
    a.tiles = rtiles * a.tok_tiles;
    const int grid = a.tiles < sm_count() ? a.tiles : sm_count();
    return launch_pdl("mmq", mmq_tc_kernel, dim3((unsigned)grid), dim3(THREADS), (size_t)SMEM_BYTES, s, a);
}

}  // namespace qk
