// Quantised-weight projections that read one shared Q8_1 activation image.
//
//   mmvq    : ordinary MUL_MAT, several projections (q/k/v, gate/up) in one
//             launch (llama.cpp PR #117 "activation image emission",
//             Overview/Coverage; its "Ordinary, K8192 / T8" component).
//   mmvq_id : routed MUL_MAT_ID over a stable expert plan; experts with no
//             planned pair read no weights (TensorFold PR #1047, "The fix").
//             Per-pair mode reads image row p for pair p (the per-slot down
//             projection; PR #117 "GLU producer evidence", per-slot routed rows).
//
// Per 32-block b of weight row n and image row t, from the stored halves:
//   Q4_0: y += d_w * (d_a * D - 8 * s_a),   D = sum nibble_i * q_i
//   Q8_0: y += d_w * (d_a * D),             D = sum w_i * q_i
//
// Block dot on the f16 tensor path. Nibbles, int8 weights and int8 codes are
// exact in binary16, products are exact and every partial sum stays below
// 2^22, so the f32 accumulator of mma.sync m16n8k16 holds the integer D
// exactly. (Blackwell Ultra's int8 mma and dp4a run at about a quarter of its
// f16 mma rate -- measured 150 vs 590 T/s -- too slow to keep up with HBM at
// 8 tokens.) A nibble becomes a half with one logic op by OR-ing it under a
// binary16 exponent (1024 + lo for low nibbles, 64 + hi for high ones); the
// bias this adds, sum_i bias * q_i, depends only on the token, so a pair of
// MMAs with a constant -bias A operand computes it once per block and it
// seeds the accumulator of all 8 row groups.
//
// Ordinary path: one persistent CTA per SM. A producer warp streams 128x128
// weight units with TMA bulk copies (cp.async.bulk, L2 evict-first) into a
// ring of shared-memory slots guarded by full/empty mbarriers; 16 consumer
// warps form four unit phases (the CTA's units with index = phase mod 4), and
// in a phase warp p does rows 32p..32p+31 of all four blocks of the unit after
// the phase's four warps have each turned one block's image words into a
// shared activation record. Work is split by equal bytes over the CTAs
// (stream-K): a row tile cut between CTAs is finished by its owner (the CTA
// holding its first unit), which adds the other CTAs' parts from a small
// caller workspace in CTA order; if they are late, the owner publishes its
// part too and the last contributor adds them, in the same order. All sums run
// in a fixed order, so results do not depend on timing or on the live-row
// count.
//
// Routed path: see mmvq_id_kernel.

#include <cstdlib>
#include <mutex>

#include "qk_internal.cuh"

namespace qk {
namespace {

__device__ unsigned int g_qk_faults = 0;

constexpr int MAX_PROJ = 8;
constexpr int VALS = UNIT_GROUPS * 4 * 32;   // accumulator values of one 128-row tile
constexpr int MAXP = 8;                      // partial sums loaded per batch
// A wait suspends the thread until the phase completes or SUSPEND_NS passes,
// and gives up after SPIN_LIMIT tries (at most about a second).
constexpr uint32_t SUSPEND_NS = 20000;
constexpr uint32_t SPIN_LIMIT = 1u << 16;
// An owner waits at most this many short sleeps for the other parts of its
// tile before taking the general path (a matter of speed, not correctness);
// the environment variable QK_MMVQ_OWNER_SPIN overrides it (0 forces the
// general path, which the tests use).
constexpr int OWNER_SPIN = 2000;

template <int WT> struct Layout;
template <> struct Layout<QK_W_Q4_0> {
    static constexpr int UNIT = Q4_UNIT_BYTES, BLOCK = Q4_BLOCK_STRIDE, SCALES = 8192, SLOTS = 16;
};
template <> struct Layout<QK_W_Q8_0> {
    static constexpr int UNIT = Q8_UNIT_BYTES, BLOCK = Q8_BLOCK_STRIDE, SCALES = 16384, SLOTS = 8;
};

struct SkProj {
    const uint8_t *w;
    float *y;
    int64_t y_stride;
    int64_t unit_base;   // first unit of this projection in the flat unit space
    int N, K, chunks, row_tiles, rt_base;
};

struct SkArgs {
    const uint8_t *img;
    int64_t img_row_bytes;
    int T;
    const int32_t *live;
    int n_proj;
    int64_t U;           // total units
    float *ws_part;      // [G][2][VALS]
    unsigned int *ws_cnt;
    int owner_spin;      // short sleeps an owner waits for the other parts (0: general path at once)
    int csplit;          // 0: stream-K; else CTAs per 128-row tile (a cluster of that size when > 1)
    SkProj p[MAX_PROJ];
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_img4(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity), "r"(SUSPEND_NS)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after SPIN_LIMIT tries, records a fault and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
    for (uint32_t i = 0; i < SPIN_LIMIT; i++)
        if (mbar_try_wait(a, parity)) return true;
    atomicOr(&g_qk_faults, 1u);
    return false;
}
// Before a producer thread leaves, every copy it issued into the ring has landed, also after
// one of its waits ran out: ring positions issued - SLOTS .. issued - 1 are the last ones of
// their slots (a barrier whose phase completed long ago passes at once). A wait that runs out
// here ends the drain; the fault is already recorded.
__device__ __forceinline__ void drain_ring(const uint64_t *full, int slots, int issued) {
    for (int x = issued > slots ? issued - slots : 0; x < issued; x++)
        if (!mbar_wait(smem_addr(full + x % slots), (uint32_t)(x / slots) & 1u)) break;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar), "l"(pol)
        : "memory");
}
// Atomic add with acquire-release semantics at GPU scope (returns the old value).
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A row tile this CTA shares with others (stream-K): where its parts live.
struct SharedTile {
    float *y;
    int64_t y_stride;
    int N, rt, R;            // rows, row tile in its projection, global row-tile index
    int c_first, c_last;     // contributing CTAs
    int first_slot;          // part slot used by c_first (later CTAs use slot 0)
};

// D = A * B + C (m16n8k16, f16 inputs, f32 accumulate); D and C may differ.
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                        const float c[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Four int8 codes (bytes c0..c3) -> exact half2 (c0, c2) and (c1, c3):
// XOR 0x80 gives u = c + 128; the half 0x64uu is 1024 + u; minus 1152 is c.
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4240);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4341);
    __half2 ha = __hsub2(as_h2(a), bias);
    __half2 hb = __hsub2(as_h2(b), bias);
    h02 = *reinterpret_cast<uint32_t *>(&ha);
    h13 = *reinterpret_cast<uint32_t *>(&hb);
}

// ---------------------------------------------------------------- one block
// Activation side of block b for this lane: B fragments of token g (elements
// 4t..4t+3 and 16+4t..16+4t+3), scales of tokens 2t and 2t+1, and the bias
// correction shared by every row group. The four image words are loaded one
// block ahead (Raw) so their latency overlaps the previous block's MMAs.
struct Raw {
    uint32_t lo, hi, ds0, ds1;
};
struct BSide {
    uint32_t lo02, lo13, hi02, hi13;
    float da0, da1, ns0, ns1;
    float corr[4];
};

__device__ __forceinline__ Raw load_raw(const uint8_t *imgB, const uint8_t *imgS0, const uint8_t *imgS1, int b,
                                        int t4) {
    Raw r = {0u, 0u, 0u, 0u};
    const uint32_t off = (uint32_t)b * Q8_1_BYTES;   // b < 2^26 (K < 2^31)
    if (imgB) {
        r.lo = ld_img4(imgB + off + 4 + 4 * t4);
        r.hi = ld_img4(imgB + off + 20 + 4 * t4);
    }
    if (imgS0) r.ds0 = ld_img4(imgS0 + off);
    if (imgS1) r.ds1 = ld_img4(imgS1 + off);
    return r;
}

template <int WT>
__device__ __forceinline__ void bside(const Raw &r, BSide &s) {
    constexpr uint32_t NEG_LO = WT == QK_W_Q4_0 ? 0xE400E400u : 0xE480E480u;  // -1024 | -1152
    constexpr uint32_t NEG_HI = WT == QK_W_Q4_0 ? 0xD400D400u : 0xE480E480u;  //   -64 | -1152
    codes_to_half2(r.lo, s.lo02, s.lo13);   // an absent token has zero words: exact zeros
    codes_to_half2(r.hi, s.hi02, s.hi13);
    const float2 d0 = __half22float2(as_h2(r.ds0)), d1 = __half22float2(as_h2(r.ds1));
    s.da0 = d0.x;
    s.da1 = d1.x;
    s.ns0 = WT == QK_W_Q4_0 ? -8.0f * d0.y : 0.0f;
    s.ns1 = WT == QK_W_Q4_0 ? -8.0f * d1.y : 0.0f;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t alo[4] = {NEG_LO, NEG_LO, NEG_LO, NEG_LO};
    const uint32_t ahi[4] = {NEG_HI, NEG_HI, NEG_HI, NEG_HI};
    float c1[4];
    mma_f16(c1, alo, s.lo02, s.lo13, zero);
    mma_f16(s.corr, ahi, s.hi02, s.hi13, c1);
}

// Block dot of one row group in a single asm block, so that the weight
// conversions write the MMA operand registers directly (built in C++, the
// operand arrays cost extra register moves):
//   D = A_lo * (lo02, lo13) + A_hi * (hi02, hi13) + C.
// Q4_0: w, w8 = nibble words of rows g and g+8 (see nibbles_to_half2).
__device__ __forceinline__ void dot_q4(uint32_t w, uint32_t w8, const BSide &s, float d[4]) {
    asm("{\n"
        ".reg .b32 s0, s1, l0, l1, l2, l3, h0, h1, h2, h3;\n"
        ".reg .f32 e0, e1, e2, e3;\n"
        "shr.b32 s0, %4, 8;\n"
        "shr.b32 s1, %5, 8;\n"
        "lop3.b32 l0, %4, 0x000F000F, 0x64006400, 0xEA;\n"
        "lop3.b32 l1, %5, 0x000F000F, 0x64006400, 0xEA;\n"
        "lop3.b32 l2, s0, 0x000F000F, 0x64006400, 0xEA;\n"
        "lop3.b32 l3, s1, 0x000F000F, 0x64006400, 0xEA;\n"
        "lop3.b32 h0, %4, 0x00F000F0, 0x54005400, 0xEA;\n"
        "lop3.b32 h1, %5, 0x00F000F0, 0x54005400, 0xEA;\n"
        "lop3.b32 h2, s0, 0x00F000F0, 0x54005400, 0xEA;\n"
        "lop3.b32 h3, s1, 0x00F000F0, 0x54005400, 0xEA;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {e0,e1,e2,e3}, {l0,l1,l2,l3}, {%6,%7}, "
        "{%10,%11,%12,%13};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {h0,h1,h2,h3}, {%8,%9}, "
        "{e0,e1,e2,e3};\n"
        "}\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(w), "r"(w8), "r"(s.lo02), "r"(s.lo13), "r"(s.hi02), "r"(s.hi13), "f"(s.corr[0]), "f"(s.corr[1]),
          "f"(s.corr[2]), "f"(s.corr[3]));
}
// Q8_0: v = one row group's 16 bytes (see the weight pack): codes of row g
// (elements 4t.. and 16+4t..) and of row g+8.
__device__ __forceinline__ void dot_q8(uint4 v, const BSide &s, float d[4]) {
    asm("{\n"
        ".reg .b32 u0, u1, u2, u3, l0, l1, l2, l3, h0, h1, h2, h3;\n"
        ".reg .f32 e0, e1, e2, e3;\n"
        "xor.b32 u0, %4, 0x80808080;\n"
        "xor.b32 u1, %5, 0x80808080;\n"
        "xor.b32 u2, %6, 0x80808080;\n"
        "xor.b32 u3, %7, 0x80808080;\n"
        "prmt.b32 l0, u0, 0x64646464, 0x4240;\n"
        "prmt.b32 l2, u0, 0x64646464, 0x4341;\n"
        "prmt.b32 h0, u1, 0x64646464, 0x4240;\n"
        "prmt.b32 h2, u1, 0x64646464, 0x4341;\n"
        "prmt.b32 l1, u2, 0x64646464, 0x4240;\n"
        "prmt.b32 l3, u2, 0x64646464, 0x4341;\n"
        "prmt.b32 h1, u3, 0x64646464, 0x4240;\n"
        "prmt.b32 h3, u3, 0x64646464, 0x4341;\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {e0,e1,e2,e3}, {l0,l1,l2,l3}, {%8,%9}, "
        "{%12,%13,%14,%15};\n"
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {h0,h1,h2,h3}, {%10,%11}, "
        "{e0,e1,e2,e3};\n"
        "}\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(s.lo02), "r"(s.lo13), "r"(s.hi02), "r"(s.hi13),
          "f"(s.corr[0]), "f"(s.corr[1]), "f"(s.corr[2]), "f"(s.corr[3]));
}

__device__ __forceinline__ void scale_epilogue(const float dv[4], uint32_t dw2, const BSide &s, float acc[4]) {
    // acc[i] += dw_row * (d_a * D + ns), the token pair's operations two at a time (fma.rn.f32x2:
    // the same correctly rounded fma per lane as fmaf, in half the issue slots)
    asm("{\n"
        ".reg .b16 hx, hy;\n"
        ".reg .f32 wx, wy;\n"
        ".reg .b64 DA, NS, D01, D23, T01, T23, WX, WY, A01, A23;\n"
        "mov.b32 {hx, hy}, %10;\n"
        "cvt.f32.f16 wx, hx;\n"
        "cvt.f32.f16 wy, hy;\n"
        "mov.b64 DA, {%6, %7};\n"
        "mov.b64 NS, {%8, %9};\n"
        "mov.b64 D01, {%4, %5};\n"
        "mov.b64 D23, {%11, %12};\n"
        "fma.rn.f32x2 T01, DA, D01, NS;\n"
        "fma.rn.f32x2 T23, DA, D23, NS;\n"
        "mov.b64 WX, {wx, wx};\n"
        "mov.b64 WY, {wy, wy};\n"
        "mov.b64 A01, {%0, %1};\n"
        "mov.b64 A23, {%2, %3};\n"
        "fma.rn.f32x2 A01, WX, T01, A01;\n"
        "fma.rn.f32x2 A23, WY, T23, A23;\n"
        "mov.b64 {%0, %1}, A01;\n"
        "mov.b64 {%2, %3}, A23;\n"
        "}\n"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3])
        : "f"(dv[0]), "f"(dv[1]), "f"(s.da0), "f"(s.da1), "f"(s.ns0), "f"(s.ns1), "r"(dw2), "f"(dv[2]), "f"(dv[3]));
}

// All 8 row groups of one block, from shared memory (SMEM, 32-bit shared
// addresses) or with streaming global loads.
template <int WT, bool SMEM>
__device__ __forceinline__ void block_rows(const uint8_t *gblk, uint32_t sblk, const uint8_t *gsc, uint32_t ssc,
                                           int lane, const BSide &s, float acc[UNIT_GROUPS][4]) {
    const int g = lane >> 2;
    uint4 sc0, sc1;
    if (SMEM) {
        sc0 = lds128(ssc + g * 32);
        sc1 = lds128(ssc + g * 32 + 16);
    } else {
        sc0 = ldg_stream16(gsc + g * 32);
        sc1 = ldg_stream16(gsc + g * 32 + 16);
    }
    const uint32_t scw[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    if (WT == QK_W_Q4_0) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint4 v = SMEM ? lds128(sblk + k * 512 + lane * 16) : ldg_stream16(gblk + k * 512 + lane * 16);
            float d0[4], d1[4];
            dot_q4(v.x, v.y, s, d0);
            dot_q4(v.z, v.w, s, d1);
            scale_epilogue(d0, scw[2 * k], s, acc[2 * k]);
            scale_epilogue(d1, scw[2 * k + 1], s, acc[2 * k + 1]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const uint4 v = SMEM ? lds128(sblk + k * 512 + lane * 16) : ldg_stream16(gblk + k * 512 + lane * 16);
            float d[4];
            dot_q8(v, s, d);
            scale_epilogue(d, scw[k], s, acc[k]);
        }
    }
}

// ---------------------------------------------------------------- ordinary path
// One persistent CTA per SM: a producer warp streams the CTA's units with TMA
// bulk copies into a ring of shared-memory slots (full/empty mbarriers), and
// 16 consumer warps work on four units at once. Warp w belongs to unit phase
// q = w >> 2 (the CTA's units with index = q mod 4) and owns row-group pair
// p = w & 3 (rows 32p..32p+31 of the 128-row tile), over all four blocks of
// each of its units, so it keeps only 2 x 4 accumulators. The activation side
// of a unit is shared through shared memory: warp (p, q) turns the image words
// of block p into an activation record (the B fragments of every lane, the
// bias-correction C operand and (d_a, -8 s_a) per pair of tokens), and the
// four warps of the phase meet at a named barrier before reading all four
// records. A slot is empty again when the phase's 128 threads have loaded
// their operands from it (each thread arrives after its own loads). At the end
// of a segment (the CTA's units of one row tile) the four phases' partial sums
// are added in fixed order.
#ifndef QK_MMVQ_PHASES
#define QK_MMVQ_PHASES 4
#endif
constexpr int NPH = QK_MMVQ_PHASES;   // units in work at once (unit phases)
constexpr int SK_CONS = 4 * NPH;
constexpr int SK_PRODUCER = SK_CONS;
constexpr int SK_THREADS = (SK_CONS + 1) * 32;
constexpr int BREC = 640;       // [0,512) fragments (16 B per lane), [512,576) C quads, [576,640) scales (per t4)
constexpr int IMG_AHEAD = 3;    // units of image words a consumer warp has in flight

static_assert(Layout<QK_W_Q4_0>::SLOTS % NPH == 0 && Layout<QK_W_Q8_0>::SLOTS % NPH == 0,
              "a ring slot must come back to the same unit phase");

template <int WT>
struct SkLayout {
    static constexpr int UNIT = Layout<WT>::UNIT, SLOTS = Layout<WT>::SLOTS;
    static constexpr int SLOT = UNIT;
    static constexpr int RECS = SLOTS * SLOT;                     // [4 phases][2][4 blocks][BREC]
    static constexpr int RED = RECS + NPH * 2 * 4 * BREC;         // [SK_CONS][256] floats
    static constexpr int KEEP = RED + SK_CONS * 256 * 4;          // [2][VALS] floats
    static constexpr int BARS = KEEP + 2 * VALS * 4;              // full[SLOTS], empty[SLOTS]
    static constexpr int BYTES = BARS + 2 * SLOTS * 8;
};

__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void all_consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(SK_CONS * 32) : "memory");
}
// The four warps of unit phase q (barriers 2..5). A warp writes its record of
// unit k into buffer k & 1 and reads all four after this barrier; it can only
// write buffer k & 1 again (unit k+2) after the barrier of unit k+1, which the
// other three warps pass only once they have read unit k's records.
__device__ __forceinline__ void phase_sync(int q) {
    asm volatile("bar.sync %0, 128;" ::"r"(2 + q) : "memory");
}

// Activation record of one block from its image words (zero words: zero record).
template <int WT>
__device__ __forceinline__ void write_record(uint32_t rec, const Raw &r, int lane) {
    BSide s;
    bside<WT>(r, s);
    sts128(rec + lane * 16, make_uint4(s.lo02, s.lo13, s.hi02, s.hi13));
    if (lane < 4) {   // lanes 0..3: g = 0, t4 = lane; the records depend on t4 only
        sts128(rec + 512 + lane * 16, make_uint4(__float_as_uint(s.corr[0]), __float_as_uint(s.corr[1]),
                                                 __float_as_uint(s.corr[2]), __float_as_uint(s.corr[3])));
        sts128(rec + 576 + lane * 16, make_uint4(__float_as_uint(s.da0), __float_as_uint(s.da1),
                                                 __float_as_uint(s.ns0), __float_as_uint(s.ns1)));
    }
}

// Row groups 2p and 2p+1 (rows 32p..32p+31) of all four blocks of the unit in
// ring slot sb: weights and scales from the unit, B operands, correction and
// token scales from the unit's four activation records at recs.
template <int WT>
__device__ __forceinline__ void unit_rows(uint32_t sb, uint32_t recs, int p, int lane, float acc[2][4]) {
    using L = Layout<WT>;
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int jb = 0; jb < 4; jb++) {
        const uint32_t rec = recs + jb * BREC;
        const uint4 bf = lds128(rec + lane * 16);
        const uint4 cq = lds128(rec + 512 + t4 * 16);
        const uint4 dq = lds128(rec + 576 + t4 * 16);
        const uint2 sc = lds64(sb + L::SCALES + jb * 256 + g * 32 + p * 8);
        BSide s;
        s.lo02 = bf.x;
        s.lo13 = bf.y;
        s.hi02 = bf.z;
        s.hi13 = bf.w;
        s.corr[0] = __uint_as_float(cq.x);
        s.corr[1] = __uint_as_float(cq.y);
        s.corr[2] = __uint_as_float(cq.z);
        s.corr[3] = __uint_as_float(cq.w);
        s.da0 = __uint_as_float(dq.x);
        s.da1 = __uint_as_float(dq.y);
        s.ns0 = __uint_as_float(dq.z);
        s.ns1 = __uint_as_float(dq.w);
        float d0[4], d1[4];
        if (WT == QK_W_Q4_0) {
            const uint4 w = lds128(sb + jb * L::BLOCK + p * 512 + lane * 16);
            dot_q4(w.x, w.y, s, d0);
            dot_q4(w.z, w.w, s, d1);
        } else {
            dot_q8(lds128(sb + jb * L::BLOCK + (2 * p) * 512 + lane * 16), s, d0);
            dot_q8(lds128(sb + jb * L::BLOCK + (2 * p + 1) * 512 + lane * 16), s, d1);
        }
        scale_epilogue(d0, sc.x, s, acc[0]);
        scale_epilogue(d1, sc.y, s, acc[1]);
    }
}

// Output position of accumulator value v (0..VALS-1) of a 128-row tile.
__device__ __forceinline__ void val_pos(int v, int &row, int &slot) {
    const int l = v & 31, i = (v >> 5) & 3, r = v >> 7;
    row = 16 * r + (l >> 2) + ((i & 2) ? 8 : 0);
    slot = 2 * (l & 3) + (i & 1);
}

__device__ __forceinline__ int64_t cta_start(int c, int64_t U, int G) {
    return (int64_t)(((uint64_t)c * (uint64_t)U) / (uint32_t)G);
}
__device__ __forceinline__ int cta_of(int64_t u, int64_t U, int G) {
    int c = (int)((u * G) / U);
    while (c + 1 < G && cta_start(c + 1, U, G) <= u) c++;
    while (c > 0 && cta_start(c, U, G) > u) c--;
    return c;
}

// Unit u of the flat unit space -> projection j, row tile rt, column chunk c.
__device__ __forceinline__ void decode_unit(const SkArgs &a, int64_t u, int &j, int &rt, int &c) {
    j = 0;
    while (j + 1 < a.n_proj && u >= a.p[j + 1].unit_base) j++;
    const uint32_t local = (uint32_t)(u - a.p[j].unit_base);   // < 2^31 units per projection
    rt = (int)(local / (uint32_t)a.p[j].chunks);
    c = (int)(local % (uint32_t)a.p[j].chunks);
}

template <int WT>
__global__ void __launch_bounds__(SK_THREADS, 1) mmvq_sk_kernel(const __grid_constant__ SkArgs a) {
    using L = Layout<WT>;
    using S = SkLayout<WT>;
    extern __shared__ __align__(128) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem + S::RED);
    float *keep = reinterpret_cast<float *>(smem + S::KEEP);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::BARS);
    uint64_t *empty = full + L::SLOTS;
    __shared__ int s_last[2];
    __shared__ SharedTile s_tile[2];

    pdl_trigger();
    const int G = gridDim.x, cta = blockIdx.x;
    int64_t u0, u1;
    int crank = 0;   // rank in the cluster (cluster split)
    if (a.csplit) {   // cluster split: CTA c takes part c % csplit of row tile c / csplit (all of K split evenly)
        const int R = cta / a.csplit;
        crank = cta % a.csplit;
        int jj = 0;
        while (jj + 1 < a.n_proj && R >= a.p[jj + 1].rt_base) jj++;
        const SkProj &P = a.p[jj];
        const int64_t first = P.unit_base + (int64_t)(R - P.rt_base) * P.chunks;
        u0 = first + (int64_t)crank * P.chunks / a.csplit;
        u1 = first + (int64_t)(crank + 1) * P.chunks / a.csplit;
    } else {
        u0 = cta_start(cta, a.U, G);
        u1 = cta_start(cta + 1, a.U, G);
    }
    const int n_units = (int)(u1 - u0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring = smem_addr(smem);
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::SLOTS; s++) {
            mbar_init(smem_addr(full + s), 1);                 // the producer, with the unit's bytes
            mbar_init(smem_addr(empty + s), 4 * 32);          // the four warps of one unit phase
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == SK_PRODUCER) {   // ---------------- producer: weights only, no wait on the previous kernel
        if (lane == 0 && n_units > 0) {
            const uint64_t pol = evict_first_policy();
            int j, rt, c;
            decode_unit(a, u0, j, rt, c);
            // units of one projection are contiguous in its packed buffer
            const uint8_t *src = a.p[j].w + ((int64_t)rt * a.p[j].chunks + c) * L::UNIT;
            int64_t left_in_proj = a.p[j].unit_base + (int64_t)a.p[j].row_tiles * a.p[j].chunks - u0;
            int issued = 0;
            for (; issued < n_units; issued++) {
                const int slot = issued % L::SLOTS;
                const uint32_t n = (uint32_t)issued / L::SLOTS;
                if (n > 0 && !mbar_wait(smem_addr(empty + slot), (n - 1) & 1u)) break;
                if (left_in_proj == 0) {   // next projection
                    j++;
                    src = a.p[j].w;
                    left_in_proj = (int64_t)a.p[j].row_tiles * a.p[j].chunks;
                }
                mbar_expect_tx(smem_addr(full + slot), L::UNIT);
                bulk_g2s(ring + (uint32_t)slot * S::SLOT, src, L::UNIT, smem_addr(full + slot), pol);
                src += L::UNIT;
                left_in_proj--;
            }
            drain_ring(full, L::SLOTS, issued);
        }
        return;
    }

    // ---------------- consumers
    int tl = 0;   // live tokens: read after the wait on the previous kernel, below
    const int tid = threadIdx.x, p = warp & 3;
    bool ok = true;

    // Row tiles this CTA shares (at most its first, slot 0, and its last, slot
    // 1), planned now so that the tail only stores, counts and adds.
    if (tid < 2) {
        SharedTile st = {};
        st.R = -1;
        if (n_units > 0 && !a.csplit) {
            int jj, rr, cc;
            decode_unit(a, tid == 0 ? u0 : u1 - 1, jj, rr, cc);
            const SkProj &P = a.p[jj];
            const int64_t rs = P.unit_base + (int64_t)rr * P.chunks, re = rs + P.chunks;
            const bool first_tile_too = tid == 1 && rs <= u0;   // last tile == first tile
            if (!first_tile_too && (rs < u0 || re > u1)) {
                st.y = P.y;
                st.y_stride = P.y_stride;
                st.N = P.N;
                st.rt = rr;
                st.R = P.rt_base + rr;
                st.c_first = cta_of(rs, a.U, G);
                st.c_last = cta_of(re - 1, a.U, G);
                st.first_slot = cta_start(st.c_first, a.U, G) < rs ? 1 : 0;
            }
        }
        s_tile[tid] = st;
    }

    all_consumers_sync();   // s_tile is planned
    // Cluster split: the leader's (rank 0) part slots, [csplit][VALS] floats after the barriers,
    // addressed through the cluster's shared-memory window.
    uint32_t cpart_leader = 0;
    if (a.csplit > 1)
        asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(cpart_leader) : "r"(ring + (uint32_t)S::BYTES));
    int signalled = 0;          // thread 0: slot + 1 of a part signalled in the loop
    unsigned signal_old = 0;

    // Sum of the parts of shared tile st in CTA order (c_first first) and the
    // store of the tile's outputs; the owner's own part comes from keep.
    auto add_parts = [&](const SharedTile &st, int ls, bool own_from_keep) {
        constexpr int PER = (VALS + SK_CONS * 32 - 1) / (SK_CONS * 32);
        float sums[PER];
#pragma unroll
        for (int k = 0; k < PER; k++) {
            const int t = tid + k * SK_CONS * 32;
            sums[k] = own_from_keep && t < VALS ? keep[ls * VALS + t] : 0.0f;
        }
        const int cfirst = own_from_keep ? st.c_first + 1 : st.c_first;
        for (int cb = cfirst; cb <= st.c_last; cb += MAXP) {   // MAXP parts in flight at once
            const float *src[MAXP];
#pragma unroll
            for (int qq = 0; qq < MAXP; qq++) {
                const int cc = cb + qq <= st.c_last ? cb + qq : st.c_last;
                const int pslot = cc == st.c_first ? st.first_slot : 0;
                src[qq] = a.ws_part + ((int64_t)cc * 2 + pslot) * VALS;
            }
#pragma unroll
            for (int k = 0; k < PER; k++) {
                const int t = tid + k * SK_CONS * 32;
                if (t >= VALS) break;
                float part[MAXP];
#pragma unroll
                for (int qq = 0; qq < MAXP; qq++) part[qq] = __ldcg(src[qq] + t);
#pragma unroll
                for (int qq = 0; qq < MAXP; qq++)
                    if (cb + qq <= st.c_last) sums[k] += part[qq];
            }
        }
#pragma unroll
        for (int k = 0; k < PER; k++) {
            const int t = tid + k * SK_CONS * 32;
            if (t >= VALS) break;
            int row, tok;
            val_pos(t, row, tok);
            row += st.rt * UNIT_ROWS;
            if (row < st.N && tok < tl) st.y[(int64_t)tok * st.y_stride + row] = sums[k];
        }
    };
    // Once this CTA's part of st is in the workspace: signal it; the
    // contributor that signals last adds all the parts. Thread 0's
    // acquire-release atomic after the barrier covers the CTA's stores.
    auto settle_part = [&](const SharedTile &st) {
        if (tid == 0) {
            const unsigned old = atom_add_acq_rel(a.ws_cnt + st.R, 1u);
            s_last[1] = old == (unsigned)(st.c_last - st.c_first);
        }
        all_consumers_sync();
        if (s_last[1]) {
            add_parts(st, 0, false);
            if (tid == 0) a.ws_cnt[st.R] = 0u;
        }
        all_consumers_sync();   // s_last is reused
    };

    int j = 0, rt = 0, c = 0;
    if (n_units > 0) decode_unit(a, u0, j, rt, c);
    const int q = warp >> 2, g = lane >> 2, t4 = lane & 3;
    const uint32_t recs_q = ring + S::RECS + (uint32_t)q * 2 * 4 * BREC;

    // The load cursor walks the phase's units (every fourth) with the current projection's sizes
    // in registers.
    int lj = j, lrt = rt, lc = c, li = q;   // cursor at this phase's first unit
    int l_kb = 0, l_chunks = 1, l_rtiles = 1;
    if (n_units > 0) {
        l_kb = a.p[lj].K / QB;
        l_chunks = a.p[lj].chunks;
        l_rtiles = a.p[lj].row_tiles;
    }
    auto cursor_step = [&](int n) {   // advance the cursor by n units
        lc += n;
        while (lc >= l_chunks) {
            lc -= l_chunks;
            if (++lrt == l_rtiles) {
                lrt = 0;
                if (++lj < a.n_proj) {
                    l_kb = a.p[lj].K / QB;
                    l_chunks = a.p[lj].chunks;
                    l_rtiles = a.p[lj].row_tiles;
                }
            }
        }
    };
    cursor_step(q);

    // Everything above depends on the arguments only and overlaps the previous kernel's tail;
    // everything below reads what that kernel wrote (image, live count, workspace) or writes
    // outputs, so it waits for it first.
    pdl_wait();
    tl = live_rows(a.live, a.T);

    // Image words of block p of this phase's units, IMG_AHEAD units ahead.
    const uint8_t *imgB = g < tl ? a.img + (int64_t)g * a.img_row_bytes : nullptr;
    const uint8_t *imgS0 = 2 * t4 < tl ? a.img + (int64_t)(2 * t4) * a.img_row_bytes : nullptr;
    const uint8_t *imgS1 = 2 * t4 + 1 < tl ? a.img + (int64_t)(2 * t4 + 1) * a.img_row_bytes : nullptr;
    auto load_next = [&]() -> Raw {   // image words of block p of unit li; then li += NPH
        Raw r = {0u, 0u, 0u, 0u};
        if (li < n_units) {
            const int b = 4 * lc + p;
            if (b < l_kb) r = load_raw(imgB, imgS0, imgS1, b, t4);
            cursor_step(NPH);
        }
        li += NPH;
        return r;
    };
    Raw img_r[IMG_AHEAD];
#pragma unroll
    for (int k = 0; k < IMG_AHEAD; k++) img_r[k] = load_next();
    int kq = 0;   // this phase's unit count so far (picks the record buffer)

    bool first_seg = true;       // the CTA's first segment keeps its part in slot 0, a later one in slot 1
    for (int i_seg = 0; i_seg < n_units;) {   // segment = this CTA's units of one row tile
        const SkProj &P = a.p[j];
        const int seg_len = P.chunks - c < n_units - i_seg ? P.chunks - c : n_units - i_seg;
        const bool whole = c == 0 && seg_len == P.chunks;
        float acc[2][4];
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int k = 0; k < 4; k++) acc[r][k] = 0.0f;
        for (int i = i_seg + ((q - i_seg) % NPH + NPH) % NPH; i < i_seg + seg_len; i += NPH, kq++) {
            // activation record of block p of this unit, from the image words loaded earlier
            const Raw cur = img_r[0];
#pragma unroll
            for (int k = 0; k + 1 < IMG_AHEAD; k++) img_r[k] = img_r[k + 1];
            img_r[IMG_AHEAD - 1] = load_next();
            const uint32_t recs = recs_q + (uint32_t)(kq & 1) * 4 * BREC;
            write_record<WT>(recs + p * BREC, cur, lane);
            phase_sync(q);   // the phase's four records are written (double buffer: see below)
            const int slot = i % L::SLOTS;
            if (ok) ok = mbar_wait(smem_addr(full + slot), ((uint32_t)i / L::SLOTS) & 1u);
            if (ok) unit_rows<WT>(ring + (uint32_t)slot * S::SLOT, recs, p, lane, acc);
            mbar_arrive(smem_addr(empty + slot));   // after this thread's shared loads
        }
        // add the four unit phases' parts in fixed order
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int k = 0; k < 4; k++) red[warp * 256 + (r * 4 + k) * 32 + lane] = acc[r][k];
        all_consumers_sync();
        const int part_slot = first_seg ? 0 : 1;
        for (int tv = tid; tv < VALS; tv += SK_CONS * 32) {
            const int pp = tv >> 8, w_in = tv & 255;
            float sum = red[pp * 256 + w_in];
#pragma unroll
            for (int qq = 1; qq < NPH; qq++) sum += red[(pp + 4 * qq) * 256 + w_in];
            if (whole) {
                int row, tok;
                val_pos(tv, row, tok);
                row += rt * UNIT_ROWS;
                if (row < P.N && tok < tl) P.y[(int64_t)tok * P.y_stride + row] = sum;
            } else if (a.csplit) {   // cluster split: into slot crank of the leader's parts
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cpart_leader + (uint32_t)(crank * VALS + tv) * 4u),
                             "f"(sum)
                             : "memory");
            } else if (cta == s_tile[part_slot].c_first) {
                keep[part_slot * VALS + tv] = sum;   // owner: kept for the end
            } else {
                __stcg(a.ws_part + ((int64_t)cta * 2 + part_slot) * VALS + tv, sum);
            }
        }
        all_consumers_sync();   // red is rewritten by the next segment
        if (!whole && !a.csplit && cta != s_tile[part_slot].c_first && tid == 0) {
            // signal the part; the result is only looked at after the loop,
            // so the atomic's latency is not waited for here
            signalled = part_slot + 1;
            signal_old = atom_add_acq_rel(a.ws_cnt + s_tile[part_slot].R, 1u);
        }
        first_seg = false;
        i_seg += seg_len;
        c = 0;                  // the next segment starts a row tile
        if (++rt == P.row_tiles) {
            rt = 0;
            j++;
        }
    }

    if (a.csplit) {
        if (a.csplit > 1) {
            // every part is in the leader's shared memory once all threads of the cluster have
            // passed this barrier (the producer warps have exited); the leader adds them in rank
            // order, and no CTA leaves while the leader may still be written
            // (the arrive releases this thread's shared::cluster stores; the wait acquires the others')
            asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
            if (crank == 0 && n_units > 0) {
                int jj, rr, cc;
                decode_unit(a, u0, jj, rr, cc);
                const SkProj &P = a.p[jj];
                const float *parts = reinterpret_cast<const float *>(smem + S::BYTES);
                for (int tv = tid; tv < VALS; tv += SK_CONS * 32) {
                    float sum = parts[tv];
                    for (int r = 1; r < a.csplit; r++) sum += parts[r * VALS + tv];
                    int row, tok;
                    val_pos(tv, row, tok);
                    row += rr * UNIT_ROWS;
                    if (ok && row < P.N && tok < tl) P.y[(int64_t)tok * P.y_stride + row] = sum;
                }
            }
        }
        return;
    }

    // A signalled part whose atomic found all the others already there: this
    // CTA adds the parts (only when the tile's owner took the general path).
    if (tid == 0) {
        s_last[1] = 0;
        if (signalled) {
            const SharedTile &st = s_tile[signalled - 1];
            s_last[1] = signal_old == (unsigned)(st.c_last - st.c_first) ? signalled : 0;
        }
    }
    all_consumers_sync();
    if (s_last[1]) {
        const SharedTile &st = s_tile[s_last[1] - 1];
        add_parts(st, 0, false);
        if (tid == 0) a.ws_cnt[st.R] = 0u;
    }

    // The owner of a shared row tile (the CTA holding its first unit; the
    // tile is its last segment) adds the other contributors' parts as soon
    // as all of them have signalled, without publishing its own. If they are
    // late it takes the general path: it publishes too, and whichever
    // contributor signals last adds all the parts.
    if (n_units > 0) {
        const int ls = s_tile[1].R >= 0 ? 1 : 0;   // slot of the last segment's tile
        const SharedTile &st = s_tile[ls];
        if (st.R >= 0 && cta == st.c_first) {
            if (tid == 0) {
                const unsigned want = (unsigned)(st.c_last - st.c_first);
                int fast = 0;
                for (int it = 0; it < a.owner_spin; it++) {
                    if (ld_acquire(a.ws_cnt + st.R) == want) {
                        fast = 1;
                        break;
                    }
                    __nanosleep(64);
                }
                s_last[0] = fast;
            }
            all_consumers_sync();
            if (s_last[0]) {
                add_parts(st, ls, true);
                if (tid == 0) a.ws_cnt[st.R] = 0u;
            } else {
                float *mine = a.ws_part + ((int64_t)cta * 2 + ls) * VALS;
                for (int t = tid; t < VALS; t += SK_CONS * 32) __stcg(mine + t, keep[ls * VALS + t]);
                all_consumers_sync();
                settle_part(st);
            }
        }
    }
}

// ---------------------------------------------------------------- routed path
// Persistent CTAs over equal work items: (live expert, pass of up to 8 of its
// planned pairs, projection, 128-row tile). Every CTA first lists the experts
// with planned pairs in ascending order, with the prefix of their pass counts
// (the same lists in every CTA), so experts without pairs form no item and
// none of their weights is read, the grid is sized once for the resident CTAs
// whatever the live count, and round-robin over items of one size balances the
// CTAs. A CTA streams its items' 128x128 units with TMA bulk copies into a
// small ring (lane 0 of a producer warp, whose lanes 1..8 fetch each later
// item's token list ahead), and RW consumer warps take the blocks: warp w
// does block w & 3 of the units with index = w >> 2 mod RW/4, for all 128 rows
// and the item's pairs. An item takes a whole number of RW/4 ring positions (a
// dummy position completes its slot without a copy), so unit u of an item
// always meets the same warps. The warps' partial sums are added in fixed warp
// order, so a row's bits depend neither on the other rows routed with it, nor
// on the live count, nor on the CTA.
constexpr int RW = 8;
constexpr int ID_PAR = RW / 4;   // units in work at once
constexpr int ID_THREADS = (RW + 1) * 32;
constexpr int ID_MAX_E = 1024;

template <int WT> struct IdLayout;
// Slot s is reused by position s + SLOTS, which must belong to the same warps
// (units in work at once divide SLOTS): a waiter two phases ahead would see
// the barrier's parity alias and pass early.
template <> struct IdLayout<QK_W_Q4_0> { static constexpr int SLOTS = 6; };
template <> struct IdLayout<QK_W_Q8_0> { static constexpr int SLOTS = 4; };
static_assert(IdLayout<QK_W_Q4_0>::SLOTS % ID_PAR == 0 && IdLayout<QK_W_Q8_0>::SLOTS % ID_PAR == 0,
              "a ring slot must come back to the same unit phase");

struct IdProj {
    const uint8_t *w;
    float *y;
    int64_t expert_bytes;
    int N, K, chunks, row_tiles, tiles_begin;   // tiles_begin: first tile of this projection within an expert
};
struct IdArgs {
    const uint8_t *img;
    int64_t img_row_bytes;
    int rows, k, n_proj, E, tiles_per_expert;
    int per_pair;   // the image has a row per pair (row p) rather than per token (row p / k)
    const int32_t *counts, *offsets, *items;
    IdProj p[MAX_PROJ];
};

template <int WT>
size_t id_smem() {
    return (size_t)IdLayout<WT>::SLOTS * Layout<WT>::UNIT + (size_t)RW * VALS * sizeof(float) +
           2 * IdLayout<WT>::SLOTS * sizeof(uint64_t) + (2 * ID_MAX_E + 1) * sizeof(int32_t);
}

__device__ __forceinline__ void id_consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(RW * 32) : "memory");
}

struct IdItem {
    int e, pass, j, rt;
};
// Item it = (global pass index) * tiles_per_expert + tile; pass_pre[l] is the
// first global pass index of live expert l (pass_pre[n_live] = all passes).
__device__ __forceinline__ IdItem id_item(const IdArgs &a, const int32_t *live_e, const int32_t *pass_pre,
                                          int n_live, int it) {
    IdItem r;
    const int gp = it / a.tiles_per_expert, q = it - gp * a.tiles_per_expert;
    int lo = 0, hi = n_live - 1;   // the last l with pass_pre[l] <= gp
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pass_pre[mid] <= gp) lo = mid;
        else hi = mid - 1;
    }
    int j = 0;
    while (j + 1 < a.n_proj && q >= a.p[j + 1].tiles_begin) j++;
    r.e = live_e[lo];
    r.pass = gp - pass_pre[lo];
    r.j = j;
    r.rt = q - a.p[j].tiles_begin;
    return r;
}

// Pair idx of expert e's planned pairs, or -1: past the expert's count, outside the items
// array (offsets not from a plan of this bucket), or not a pair of this bucket.
__device__ __forceinline__ int plan_pair(const IdArgs &a, int e, int idx) {
    const int n_items = __ldg(a.counts + e);
    const int64_t at = (int64_t)__ldg(a.offsets + e) + idx;
    if (idx >= n_items || at < 0 || at >= (int64_t)a.rows * a.k) return -1;
    const int p = __ldg(a.items + at);
    return p < 0 || p / a.k >= a.rows ? -1 : p;
}

template <int WT>
__global__ void __launch_bounds__(ID_THREADS, 2) mmvq_id_kernel(const __grid_constant__ IdArgs a) {
    using L = Layout<WT>;
    constexpr int SLOTS = IdLayout<WT>::SLOTS;
    extern __shared__ __align__(128) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem + SLOTS * L::UNIT);   // [RW][VALS]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + RW * VALS);
    uint64_t *empty = full + SLOTS;
    int32_t *live_e = reinterpret_cast<int32_t *>(empty + SLOTS);   // [ID_MAX_E]
    int32_t *pass_pre = live_e + ID_MAX_E;                            // [ID_MAX_E + 1]
    // token lists of the CTA's items, double-buffered by item parity: the consumers read the first
    // item's themselves; lanes 1..8 of the producer warp write item k's (k >= 1) into buffer k & 1
    // while item k - 1 runs (meta_full), and the consumers release a buffer after its item (meta_empty)
    __shared__ int tok_img[2][8], tok_out[2][8], w_live[RW + 1], w_pass[RW + 1];
    __shared__ __align__(8) uint64_t meta_full[2], meta_empty[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t4 = lane & 3, g = lane >> 2;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; s++) {
            mbar_init(smem_addr(full + s), 1);
            mbar_init(smem_addr(empty + s), 4 * 32);   // the four warps that take a unit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(smem_addr(meta_full + b), 8);   // the eight token-list lanes
            mbar_init(smem_addr(meta_empty + b), 1);  // the consumers, once the item is stored
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_trigger();
    pdl_wait();   // counts, offsets and items come from the plan kernel
    // The experts with planned pairs, ascending, and the prefix of their pass counts. Warp w
    // takes a contiguous run of 32-expert chunks: it counts its run, the runs are prefixed over
    // warps, and the run is walked again to write its entries.
    const int nch = (a.E + 31) / 32, cpw = (nch + RW) / (RW + 1);
    const int c_begin = warp * cpw, c_end = min(nch, c_begin + cpw);
    const unsigned lt = (1u << lane) - 1u;
    auto expert_at = [&](int c, int &e, int &passes) {
        e = 32 * c + lane;
        // a count outside [0, rows * k] (not from a plan of this bucket) is clamped, so the work
        // stays bounded; plan_pair keeps every read inside items
        const int cnt = e < a.E ? min(max(__ldg(a.counts + e), 0), a.rows * a.k) : 0;
        passes = cnt > 0 ? (cnt + 7) / 8 : 0;
    };
    {
        int nl = 0, np = 0;
        for (int c = c_begin; c < c_end; c++) {
            int e, ps;
            expert_at(c, e, ps);
            nl += __popc(__ballot_sync(0xffffffffu, ps > 0));
            np += (int)__reduce_add_sync(0xffffffffu, (unsigned)ps);
        }
        if (lane == 0) {
            w_live[warp] = nl;
            w_pass[warp] = np;
        }
    }
    __syncthreads();
    {
        int bl = 0, bp = 0;
        for (int w = 0; w < warp; w++) {
            bl += w_live[w];
            bp += w_pass[w];
        }
        for (int c = c_begin; c < c_end; c++) {
            int e, ps;
            expert_at(c, e, ps);
            const unsigned m = __ballot_sync(0xffffffffu, ps > 0);
            int incl = ps;   // inclusive scan of the pass counts over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (ps > 0) {
                const int l = bl + __popc(m & lt);
                live_e[l] = e;
                pass_pre[l] = bp + incl - ps;
            }
            bl += __popc(m);
            bp += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (warp == RW && lane == 0) pass_pre[bl] = bp;   // the last warp's run ends the list
    }
    __syncthreads();
    int n_live = 0;
    for (int w = 0; w <= RW; w++) n_live += w_live[w];
    // No plan of this bucket has more passes than ceil(rows * k / 8) + (experts with pairs); a
    // larger (or wrapped) total means counts that are not a plan: no work, and bit 1 of the
    // fault word. The host keeps that bound times tiles_per_expert below 2^31.
    const int64_t tot = n_live > 0 ? pass_pre[n_live] : 0;
    const bool plan_ok = tot >= 0 && tot <= ((int64_t)a.rows * a.k + 7) / 8 + n_live;
    if (!plan_ok && threadIdx.x == 0) atomicOr(&g_qk_faults, 2u);
    const int n_work = plan_ok ? (int)tot * a.tiles_per_expert : 0, G = gridDim.x;
    const uint32_t ring = smem_addr(smem);

    if (warp == RW) {   // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = evict_first_policy();
            uint32_t pos = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_work && ok; it += G) {
                const IdItem w = id_item(a, live_e, pass_pre, n_live, it);
                const IdProj &P = a.p[w.j];
                const int pp = (P.chunks + ID_PAR - 1) / ID_PAR * ID_PAR;
                const uint8_t *wbase = P.w + (int64_t)w.e * P.expert_bytes + (int64_t)w.rt * P.chunks * L::UNIT;
                for (int u = 0; u < pp && ok; u++, pos++) {
                    const int slot = pos % SLOTS;
                    const uint32_t n = pos / SLOTS;
                    if (n > 0 && !mbar_wait(smem_addr(empty + slot), (n - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    if (u < P.chunks) {
                        mbar_expect_tx(smem_addr(full + slot), L::UNIT);
                        bulk_g2s(ring + (uint32_t)slot * L::UNIT, wbase + (int64_t)u * L::UNIT, L::UNIT,
                                 smem_addr(full + slot), pol);
                    } else {
                        mbar_arrive(smem_addr(full + slot));   // dummy position: completes the phase
                    }
                }
            }
            drain_ring(full, SLOTS, (int)pos);
        } else if (lane <= 8) {   // lanes 1..8: slot lane - 1 of the token list of items 1, 2, ... ahead
            const int q = lane - 1;
            int k = 1;
            for (int it = blockIdx.x + G; it < n_work; it += G, k++) {
                const int b = k & 1;
                if (k >= 2 && !mbar_wait(smem_addr(meta_empty + b), ((k >> 1) - 1) & 1u)) break;
                const IdItem w = id_item(a, live_e, pass_pre, n_live, it);
                const int p = plan_pair(a, w.e, w.pass * 8 + q);
                tok_img[b][q] = p >= 0 ? (a.per_pair ? p : p / a.k) : -1;
                tok_out[b][q] = p;
                mbar_arrive(smem_addr(meta_full + b));
            }
        }
        return;
    }

    // ---------------- consumers
    bool ok = true;
    const int jb = warp & 3, par = warp >> 2;
    uint32_t pos0 = 0;   // ring position of the current pass's first unit
    int k = 0;           // this CTA's item count so far (picks the token-list buffer)
    for (int it = blockIdx.x; it < n_work; it += G, k++) {
        const IdItem w = id_item(a, live_e, pass_pre, n_live, it);
        const IdProj &P = a.p[w.j];
        const int Kb = P.K / QB, chunks = P.chunks;
        const int pp = (chunks + ID_PAR - 1) / ID_PAR * ID_PAR;
        const int mb = k & 1;
        if (k == 0) {   // the first item's token list: no earlier item to hide its loads behind
            if (threadIdx.x < 8) {
                const int p = plan_pair(a, w.e, w.pass * 8 + threadIdx.x);
                tok_img[0][threadIdx.x] = p >= 0 ? (a.per_pair ? p : p / a.k) : -1;
                tok_out[0][threadIdx.x] = p;
            }
            id_consumers_sync();
        } else if (ok) {   // later items': prefetched; buffer 1 holds items 1, 3, ..., buffer 0 items 2, 4, ...
            const uint32_t phase = (k & 1) ? (uint32_t)(k >> 1) : (uint32_t)((k >> 1) - 1);
            ok = mbar_wait(smem_addr(meta_full + mb), phase & 1u);
        }
        {
            const int rB = tok_img[mb][g], rS0 = tok_img[mb][2 * t4], rS1 = tok_img[mb][2 * t4 + 1];
            const uint8_t *imgB = rB >= 0 ? a.img + (int64_t)rB * a.img_row_bytes : nullptr;
            const uint8_t *imgS0 = rS0 >= 0 ? a.img + (int64_t)rS0 * a.img_row_bytes : nullptr;
            const uint8_t *imgS1 = rS1 >= 0 ? a.img + (int64_t)rS1 * a.img_row_bytes : nullptr;
            float acc[UNIT_GROUPS][4];
#pragma unroll
            for (int r = 0; r < UNIT_GROUPS; r++)
#pragma unroll
                for (int i = 0; i < 4; i++) acc[r][i] = 0.0f;
            // this warp's units: u = par mod ID_PAR; the image words one unit ahead
            int u = par;
            Raw next = {0u, 0u, 0u, 0u};
            if (u < chunks && 4 * u + jb < Kb) next = load_raw(imgB, imgS0, imgS1, 4 * u + jb, t4);
            for (; u < pp; u += ID_PAR) {
                const Raw cur = next;
                if (u + ID_PAR < chunks && 4 * (u + ID_PAR) + jb < Kb)
                    next = load_raw(imgB, imgS0, imgS1, 4 * (u + ID_PAR) + jb, t4);
                const uint32_t pos = pos0 + u;
                const int slot = pos % SLOTS;
                if (ok) ok = mbar_wait(smem_addr(full + slot), (pos / SLOTS) & 1u);
                if (ok && u < chunks && 4 * u + jb < Kb) {
                    BSide bs;
                    bside<WT>(cur, bs);
                    const uint32_t ub = ring + (uint32_t)slot * L::UNIT;
                    block_rows<WT, true>(nullptr, ub + jb * L::BLOCK, nullptr, ub + L::SCALES + jb * 256, lane, bs,
                                         acc);
                }
                mbar_arrive(smem_addr(empty + slot));   // after this thread's shared loads
            }
#pragma unroll
            for (int r = 0; r < UNIT_GROUPS; r++)
#pragma unroll
                for (int i = 0; i < 4; i++) red[warp * VALS + (r * 4 + i) * 32 + lane] = acc[r][i];
            id_consumers_sync();
            for (int t = threadIdx.x; t < VALS; t += RW * 32) {
                float sum = 0.0f;
#pragma unroll
                for (int ww = 0; ww < RW; ww++) sum += red[ww * VALS + t];
                int row, slot;
                val_pos(t, row, slot);
                row += w.rt * UNIT_ROWS;
                const int orow = tok_out[mb][slot];
                if (row < P.N && orow >= 0) P.y[(int64_t)orow * P.N + row] = sum;
            }
            id_consumers_sync();   // red is reused by the next item, the token list two items on
            if (threadIdx.x == 0) mbar_arrive(smem_addr(meta_empty + mb));
        }
        pos0 += pp;
    }
}

// ---------------------------------------------------------------- wait self-test
// One warp waits, with the bounded wait every kernel here uses, on a
// shared-memory barrier that nothing completes: the wait runs out (about a
// second at most), sets bit 0 of the fault word and the kernel returns, so the
// failure path can be checked on a device without faulting it.
__global__ void __launch_bounds__(32) wait_selftest_kernel() {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0u);   // no thread ever arrives
}

// ---------------------------------------------------------------- weight pack
// One CTA of 256 threads per 128x128 unit. Canonical blocks are only 2-byte
// aligned, so they are read byte by byte.
template <int WT>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ src, int N, int K, int chunks,
                                                   uint8_t *__restrict__ dst) {
    using L = Layout<WT>;
    constexpr int SB = WT == QK_W_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES;
    constexpr int REGIONS = WT == QK_W_Q4_0 ? 4 : 8;
    const int64_t unit = blockIdx.x;
    const int rt = (int)(unit / chunks), c = (int)(unit % chunks);
    const int Kb = K / QB;
    uint8_t *out = dst + unit * L::UNIT;
    auto byte_at = [&](int n, int b, int off) -> uint32_t {
        if (n >= N || b >= Kb) return 0u;
        return src[((int64_t)n * Kb + b) * SB + off];
    };
    auto word_at = [&](int n, int b, int off) -> uint32_t {
        return byte_at(n, b, off) | (byte_at(n, b, off + 1) << 8) | (byte_at(n, b, off + 2) << 16) |
               (byte_at(n, b, off + 3) << 24);
    };
    const int n0 = rt * UNIT_ROWS;
    for (int idx = threadIdx.x; idx < 4 * REGIONS * 32; idx += 256) {
        const int jb = idx / (REGIONS * 32), k = (idx / 32) % REGIONS, l = idx % 32, g = l >> 2, t = l & 3;
        const int b = 4 * c + jb;
        uint4 v;
        if (WT == QK_W_Q4_0) {
            const int off = 2 + 4 * t;
            v.x = word_at(n0 + 32 * k + g, b, off);
            v.y = word_at(n0 + 32 * k + g + 8, b, off);
            v.z = word_at(n0 + 32 * k + 16 + g, b, off);
            v.w = word_at(n0 + 32 * k + 24 + g, b, off);
        } else {
            v.x = word_at(n0 + 16 * k + g, b, 2 + 4 * t);
            v.y = word_at(n0 + 16 * k + g, b, 18 + 4 * t);
            v.z = word_at(n0 + 16 * k + g + 8, b, 2 + 4 * t);
            v.w = word_at(n0 + 16 * k + g + 8, b, 18 + 4 * t);
        }
        *reinterpret_cast<uint4 *>(out + jb * L::BLOCK + k * 512 + l * 16) = v;
    }
    // scales: block jb, lane group g, row group r -> half2 (row 16r+g, row 16r+g+8)
    for (int idx = threadIdx.x; idx < 4 * 8 * 8; idx += 256) {
        const int jb = idx / 64, g = (idx / 8) % 8, r = idx % 8;
        const int b = 4 * c + jb, n = n0 + 16 * r + g;
        const uint32_t lo = byte_at(n, b, 0) | (byte_at(n, b, 1) << 8);
        const uint32_t hi = byte_at(n + 8, b, 0) | (byte_at(n + 8, b, 1) << 8);
        *reinterpret_cast<uint32_t *>(out + L::SCALES + jb * 256 + g * 32 + r * 4) = lo | (hi << 16);
    }
}

}  // namespace

int sm_count() {
    constexpr int MAXDEV = 64;
    static int n[MAXDEV] = {};   // per device: the grid sizes and workspace layout depend on it
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAXDEV) return 148;
    if (n[dev] <= 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n[dev] = v;
    }
    return n[dev];
}

namespace {

template <int WT>
size_t sk_smem() {
    using L = Layout<WT>;
    return (size_t)SkLayout<WT>::BYTES;
}

}  // namespace

// Workspace of the ordinary path: [G][2][VALS] partial sums, then one counter
// per 128-row tile; G = min(units, SMs) CTAs.
int64_t mmvq_workspace_bytes(int n_proj, const qk_proj *projs) {
    int64_t off = 0, bytes = 0;
    mmvq_counter_range(n_proj, projs, &off, &bytes);
    return off + bytes;
}

void mmvq_counter_range(int n_proj, const qk_proj *projs, int64_t *offset, int64_t *bytes) {
    int64_t U = 0, R = 0;
    for (int j = 0; j < n_proj; j++) {
        const int64_t rts = ceil_div(projs[j].N, UNIT_ROWS);
        U += rts * ceil_div(projs[j].K, UNIT_COLS);
        R += rts;
    }
    const int64_t G = U < sm_count() ? U : sm_count();
    *offset = G * 2 * VALS * (int64_t)sizeof(float);
    *bytes = R * (int64_t)sizeof(unsigned int);
}

qk_status launch_wait_selftest(cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>();
    count_launch();
    return check_launch("wait_selftest");
}

qk_status read_device_faults(uint32_t *faults) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_qk_faults, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_qk_faults, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "qk_device_faults: %s", cudaGetErrorString(e));
    *faults = v;
    return QK_OK;
}

qk_status launch_weight_pack(int wtype, const uint8_t *blocks, int64_t N, int64_t K, uint8_t *packed,
                             cudaStream_t s) {
    const int64_t chunks = ceil_div(K, UNIT_COLS);
    const int64_t units = ceil_div(N, UNIT_ROWS) * chunks;
    if (units == 0) return QK_OK;
    if (wtype == QK_W_Q4_0)
        pack_kernel<QK_W_Q4_0><<<(unsigned)units, 256, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    else
        pack_kernel<QK_W_Q8_0><<<(unsigned)units, 256, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    count_launch();
    return check_launch("weight_pack");
}

template <int WT>
static qk_status configure_sk() {
    static bool configured = false;
    if (!configured) {
        // room for the cluster split's part slots (up to 8 x VALS floats) after the stream-K layout
        const int smem = (int)(sk_smem<WT>() + 8 * VALS * sizeof(float));
        cudaError_t e = cudaFuncSetAttribute(mmvq_sk_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return fail(QK_ERR_CUDA, "mmvq: shared memory attribute: %s", cudaGetErrorString(e));
        configured = true;
    }
    return QK_OK;
}

template <int WT>
static qk_status launch_sk(const SkArgs &a, int G, cudaStream_t s) {
    qk_status st = configure_sk<WT>();
    if (st != QK_OK) return st;
    const int cl = a.csplit > 1 ? a.csplit : 1;
    const size_t smem = sk_smem<WT>() + (cl > 1 ? (size_t)cl * VALS * sizeof(float) : 0);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(SK_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cl > 1 ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mmvq_sk_kernel<WT>, a);
    count_launch();
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "mmvq: %s", cudaGetErrorString(e));
    return check_launch("mmvq");
}

// Clusters of `cl` CTAs of the ordinary kernel that can be resident at once on the current
// device (cached per device; -1 when the query fails, so the cluster split is not used).
template <int WT>
static int sk_max_clusters(int cl) {
    constexpr int MAXDEV = 64;
    static int cache[MAXDEV][9] = {};
    int dev = 0;
    if (cl < 2 || cl > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAXDEV) return -1;
    int &v = cache[dev][cl];
    if (v == 0) {
        if (configure_sk<WT>() != QK_OK) return -1;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(cl * 64);
        cfg.blockDim = dim3(SK_THREADS);
        cfg.dynamicSmemBytes = sk_smem<WT>() + (size_t)cl * VALS * sizeof(float);
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mmvq_sk_kernel<WT>, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = -1;
        }
        v = n;
    }
    return v;
}

qk_status launch_mmvq(const uint8_t *img, int64_t row_blocks, int T, int n_proj, const qk_proj *projs,
                      const int32_t *live, void *ws, size_t ws_bytes, cudaStream_t s) {
    SkArgs a = {};
    a.img = img;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.T = T;
    a.live = live;
    a.n_proj = n_proj;
    int64_t U = 0;
    int R = 0;
    for (int j = 0; j < n_proj; j++) {
        SkProj &d = a.p[j];
        d.w = static_cast<const uint8_t *>(projs[j].w);
        d.y = projs[j].y;
        d.y_stride = projs[j].y_stride;
        d.N = (int)projs[j].N;
        d.K = (int)projs[j].K;
        d.chunks = (int)ceil_div(d.K, UNIT_COLS);
        d.row_tiles = (int)ceil_div(d.N, UNIT_ROWS);
        d.unit_base = U;
        d.rt_base = R;
        U += (int64_t)d.row_tiles * d.chunks;
        R += d.row_tiles;
    }
    a.U = U;
    static const int owner_spin = [] {
        const char *e = getenv("QK_MMVQ_OWNER_SPIN");
        return e ? atoi(e) : OWNER_SPIN;
    }();
    a.owner_spin = owner_spin;
    int G = (int)(U < sm_count() ? U : sm_count());
    const int64_t need = mmvq_workspace_bytes(n_proj, projs);
    if (!ws || ws_bytes < (size_t)need)
        return fail(QK_ERR_WORKSPACE, "mmvq: workspace %zu < %lld bytes", ws_bytes, (long long)need);
    a.ws_part = static_cast<float *>(ws);
    a.ws_cnt = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(ws) + (int64_t)G * 2 * VALS * sizeof(float));
    // Cluster split instead of stream-K when the row tiles map onto the SMs in one wave of
    // clusters of at most 4 CTAs (csplit CTAs per tile, each a contiguous part of K) and no CTA
    // then takes more units than its stream-K share: the tile's parts are added through the
    // leader's shared memory instead of the workspace and L2 (q/k/v: 36 tiles x 4 CTAs, 7 units
    // each). Measured: 5-CTA clusters over the 18944 -> 3584 down projection (30 units per CTA
    // instead of 28) ran 44% slower than stream-K, so larger clusters and longer ranges are not used.
    const bool q4 = projs[0].wtype == QK_W_Q4_0;
    int cmin = 1 << 30;
    for (int j = 0; j < n_proj; j++) cmin = a.p[j].chunks < cmin ? a.p[j].chunks : cmin;
    int cs = R > 0 ? sm_count() / R : 0;
    cs = cs > 4 ? 4 : cs;
    cs = cs > cmin ? cmin : cs;
    if (cs >= 1) {
        int cmax = 0;
        for (int j = 0; j < n_proj; j++) cmax = a.p[j].chunks > cmax ? a.p[j].chunks : cmax;
        const int64_t per_cluster_cta = ceil_div(cmax, cs), per_sk_cta = ceil_div(U, G);
        const int fit = cs == 1 ? sm_count() : (q4 ? sk_max_clusters<QK_W_Q4_0>(cs) : sk_max_clusters<QK_W_Q8_0>(cs));
        if (per_cluster_cta <= per_sk_cta && fit >= R) {
            a.csplit = cs;
            G = R * cs;
        }
    }
    return q4 ? launch_sk<QK_W_Q4_0>(a, G, s) : launch_sk<QK_W_Q8_0>(a, G, s);
}

qk_status launch_mmvq_id(const uint8_t *img, int64_t row_blocks, int rows, int k, int n_proj,
                         const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                         const int32_t *items, bool per_pair, cudaStream_t s) {
    IdArgs a = {};
    a.img = img;
    a.per_pair = per_pair ? 1 : 0;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.rows = rows;
    a.k = k;
    a.n_proj = n_proj;
    a.E = (int)projs[0].n_experts;
    a.counts = counts;
    a.offsets = offsets;
    a.items = items;
    int tiles = 0;
    for (int j = 0; j < n_proj; j++) {
        IdProj &d = a.p[j];
        d.w = static_cast<const uint8_t *>(projs[j].w);
        d.y = projs[j].y;
        d.expert_bytes = packed_bytes(projs[j].wtype, projs[j].N, projs[j].K);
        d.N = (int)projs[j].N;
        d.K = (int)projs[j].K;
        d.chunks = (int)ceil_div(d.K, UNIT_COLS);
        d.row_tiles = (int)ceil_div(d.N, UNIT_ROWS);
        d.tiles_begin = tiles;
        tiles += d.row_tiles;
    }
    a.tiles_per_expert = tiles;
    if (a.E > ID_MAX_E) return fail(QK_ERR_UNSUPPORTED, "mmvq_id: n_experts=%d > %d", a.E, ID_MAX_E);
    const bool q4 = projs[0].wtype == QK_W_Q4_0;
    auto kernel = q4 ? mmvq_id_kernel<QK_W_Q4_0> : mmvq_id_kernel<QK_W_Q8_0>;
    const size_t smem = q4 ? id_smem<QK_W_Q4_0>() : id_smem<QK_W_Q8_0>();
    static int per_sm[2] = {0, 0};   // resident CTAs per SM, after the shared-memory attribute
    int &occ = per_sm[q4 ? 0 : 1];
    if (occ == 0) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, ID_THREADS, smem);
        if (e != cudaSuccess || occ < 1)
            return fail(QK_ERR_CUDA, "mmvq_id: kernel configuration: %s", cudaGetErrorString(e));
    }
    const int64_t work_max = (int64_t)a.E * tiles;
    const int64_t resident = (int64_t)occ * sm_count();
    const int G = (int)(work_max < resident ? work_max : resident);
    return launch_pdl("mmvq_id", kernel, dim3((unsigned)G), dim3(ID_THREADS), smem, s, a);
}

}  // namespace qk

// ------------------------------------------------------------------ no-allocation variant
// qk_mmvq_static_ws: the workspace is this file-scope device array instead of
// caller memory. In host code the array's name is only a host-side stand-in,
// so its device address is looked up once per device (with that device
// current) and cached.
static __device__ __align__(256) unsigned char g_mmvq_static_ws[QK_MMVQ_STATIC_WS_BYTES];

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_static_ws_mu;
void *g_static_ws_ptr[MAX_DEVICES] = {};
}  // namespace

extern "C" QK_API qk_status qk_mmvq_static_ws(const void *img, int64_t img_row_blocks, int64_t T,
                                              int32_t n_proj, const qk_proj *projs,
                                              const int32_t *d_live_rows, qk_stream stream) {
    // Every argument is checked before anything is enqueued, as in qk_mmvq.
    qk_status st = qk::mmvq_validate(img, img_row_blocks, T, n_proj, projs);
    if (st != QK_OK) return st;
    const size_t need = qk_mmvq_workspace_bytes(n_proj, projs);
    if (need > QK_MMVQ_STATIC_WS_BYTES)
        return qk::fail(QK_ERR_UNSUPPORTED, "qk_mmvq_static_ws: needs %zu bytes of scratch, the static array holds %u",
                        need, (unsigned)QK_MMVQ_STATIC_WS_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES) return qk::fail(QK_ERR_UNSUPPORTED, "qk_mmvq_static_ws: device %d", dev);
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_ws_mu);
        if (!g_static_ws_ptr[dev]) {
            e = cudaGetSymbolAddress(&g_static_ws_ptr[dev], g_mmvq_static_ws);
            if (e != cudaSuccess) {
                g_static_ws_ptr[dev] = nullptr;
                return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            }
        }
        ws = g_static_ws_ptr[dev];
    }
    // Only the completion counters must start at zero: every launch returns them to
    // zero itself, so this clear matters after a bounded wait ran out and left one
    // set. The partial-sum slots are always written before they are read. One
    // launch per weight type present, so one counter range per type.
    for (int wt = QK_W_Q4_0; wt <= QK_W_Q8_0; wt++) {
        qk_proj group[8];
        int n = 0;
        for (int j = 0; j < n_proj; j++)
            if (projs[j].wtype == wt) group[n++] = projs[j];
        if (n == 0) continue;
        int64_t off = 0, bytes = 0;
        qk::mmvq_counter_range(n, group, &off, &bytes);
        e = cudaMemsetAsync(static_cast<unsigned char *>(ws) + off, 0, (size_t)bytes, (cudaStream_t)stream);
        if (e != cudaSuccess)
            return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: clearing the counters: %s", cudaGetErrorString(e));
    }
    return qk_mmvq(img, img_row_blocks, T, n_proj, projs, d_live_rows, ws, QK_MMVQ_STATIC_WS_BYTES, stream);
}
