// kvq_prefill.cuh -- attention over the quantized cache for long query chunks
// (chunked prefill) on the sm_103a tensor cores (tcgen05, accumulators in TMEM).
//
// One CTA = (row tile, split s, kv head h, sequence b) of a work group: it
// attends kPM = 128 query rows of kv head h (row g = query token g / group,
// query head grp_q[g % group]) over split s's positions of sequence b ([0,
// chunk0) for s = 0, then chunk-sized pieces), 64 positions (one KV tile) at a
// time, and writes the final output (one split) or a partial (normalised o,
// lse) for the combine kernel.  CTAs are ordered like the split kernel's, or
// split first when the launch is split unevenly (large first pieces ahead).
//
// What it computes is the split kernel's arithmetic (scheme of the quantized
// KV cache pages: per-32 int8 K and Q with fp16 scales, integer block dot,
// q4_0 / q8_0 V), laid out for a 128-row MMA:
//   * Q codes (int8 rule, fp16 scale per 32-block) and K codes enter the MMA as
//     exact fp16 integers; per 32-block b one accumulator S_b = Q_b K_b^T (two
//     K = 16 steps) in TMEM, exact since every partial sum is an integer below
//     2^24.  score = sum_b S_b * (sq_b * sm_scale * log2 e) * sk_b.
//   * online softmax in base 2, one thread per query row (its TMEM lane), with
//     the row's reference max raised only when a score passes it by more than
//     3 (p <= 8); the P.V accumulator in TMEM is rescaled on those tiles.
//   * P.V: V is dequantized once per tile for all 128 rows, v = d * code
//     (exact in fp32), and each of p and v/2 is split into an fp16 high part
//     and an fp16 low part; O += P_hi V_hi + P_lo V_hi + P_hi V_lo keeps ~22
//     bits of every product.  (The 1/2 keeps d * code inside fp16's range
//     when the q8_0 scale rounded up; it is undone at the end.)
//
// Warp roles (512 threads, one CTA per SM, all 512 TMEM columns):
//   warps 0-7   softmax: two per TMEM lane quarter (positions 0-31 / 32-63 of
//               a tile); Q quantization into TMEM, score assembly from the
//               four S_b, softmax, P (hi, lo) into TMEM, O rescale and the
//               final O read-out;
//   warps 8-9   K converters: K codes to the fp16 operand layout, K scales,
//               the slot records;
//   warps 10-13 V converters: V codes to v/2 hi and lo;
//   warp 14     QK issuer (and the TMEM allocation);
//   warp 15     P.V issuer; it also walks the segments and issues the bulk
//               copies of the raw tiles, three stages ahead.
// The issuers run their loops as converged warps and issue every MMA, commit
// and copy from one lane elected inside the instruction's asm.  QK(j+1) is
// issued once K(j+1) is converted and the softmax has read S(j); P.V(j) once
// P(j) is in TMEM and V(j) converted, so the tensor core computes the next
// scores while the softmax works on the current ones.  Every wait suspends
// the warp (try_wait) and is bounded: a wait that gives up marks the CTA, the
// roles leave their loops, in-flight copies and MMAs are waited for (bounded),
// TMEM is released and the CTA's rows are written as NaN.
//
// Operands live in shared memory, K-major without swizzle: 8 rows x 16 bytes
// core matrices, a row group's core matrices LBO bytes apart along K (128 for
// V, 160 for K, see PrefillCfg) and row groups SBO bytes apart.
//
// The DUMP flavour (test hook) runs the same pipeline and, instead of out and
// lse, writes each row's quantized query (codes and fp16 scales) and the raw
// block accumulators S_b it reads from tensor memory, as int32, for every
// visible position of the split: the integer block dots as this kernel's
// tensor cores computed them.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kPM = kPrefillRows;        // query rows per CTA (MMA M, TMEM lanes): 128
constexpr int kPN = kPrefillPositions;   // positions per KV tile: 64
constexpr int kPSub = kPN / kWTile;      // cache tiles per KV tile (4)
constexpr int kPSoftWarps = 8;              // two per TMEM lane quarter: positions 0-31 / 32-63
constexpr int kPKWarp0 = kPSoftWarps;       // two K converter warps
constexpr int kPVWarp0 = kPKWarp0 + 2;      // four V converter warps
constexpr int kPCtlWarp = kPVWarp0 + 4;     // QK MMAs
constexpr int kPPvWarp = kPCtlWarp + 1;     // P.V MMAs and the bulk copies
constexpr int kPWarps = kPPvWarp + 1;
constexpr int kPThreads = kPWarps * 32;
constexpr float kPVScale = 0.5f;         // V enters the MMA as v / 2

template <int VT>
struct PrefillCfg {
    static constexpr int VCODE = (VT == KVQ_V_Q4_0) ? kD / 2 : kD;
    static constexpr int TILE_K = kWTile * kD, TILE_S = kWTile * kNB * 2, TILE_V = kWTile * VCODE;
    static constexpr int TILE = TILE_K + TILE_S + TILE_V + TILE_S;
    static constexpr int RS = 3;                                     // raw stages
    // raw stage: up to kPSub consecutive cache tiles of one segment piece,
    // each array's tiles side by side as in the cache
    static constexpr int R_K = 0, R_KS = R_K + kPSub * TILE_K, R_V = R_KS + kPSub * TILE_S;
    static constexpr int R_VS = R_V + kPSub * TILE_V, RAW = R_VS + kPSub * TILE_S;
    // operands (bytes)
    // K operand: 8-position row groups of 16 core matrices (8 positions x 8
    // dims, 128 bytes each) along the dims, K_LBO apart: 160 rather than 128
    // so that an 8-lane phase of a converter warp (positions 0..1 x four dim
    // groups) stores to eight distinct 16-byte bank groups
    static constexpr int K_LBO = 160;
    static constexpr int K_SBO = 16 * K_LBO;                         // 128 dims per row group
    static constexpr int KBUF = (kPN / 8) * K_SBO;                   // one K operand (64 positions)
    static constexpr int V_SBO = (kPN / 8) * 128 + 16;               // 64 positions per row group, padded so that the
                                                                     // converters' stores hit distinct banks
    static constexpr int K_OFF = 0;                                  // [2] K operands [64 positions][128 dims]
    static constexpr int VBUF = (kD / 8) * V_SBO;                    // [128 dims][64 positions]
    static constexpr int VH_OFF = K_OFF + 2 * KBUF;                  // [2] V buffers
    static constexpr int VL_OFF = VH_OFF + 2 * VBUF;
    static constexpr int RAW_OFF = VL_OFF + 2 * VBUF;
    static constexpr int SKF_OFF = RAW_OFF + RS * RAW;               // fp32 [2][block][64 positions]
    static constexpr int REC_OFF = SKF_OFF + 2 * kNB * kPN * 4;      // int4 [RS][kPSub] (tb, la, le, pos)
    static constexpr int NSUB_OFF = REC_OFF + RS * kPSub * 16;       // int [RS]
    static constexpr int OREC_OFF = (NSUB_OFF + RS * 4 + 15) / 16 * 16;   // int4 [2][kPSub]
    static constexpr int ONSUB_OFF = OREC_OFF + 2 * kPSub * 16;      // int [2]
    static constexpr int QSL_OFF = (ONSUB_OFF + 8 + 15) / 16 * 16;   // fp32 [128 rows][block]: query scales
    static constexpr int XM_OFF = QSL_OFF + kPM * kNB * 4;           // fp32 [tile parity][half][128]: tile maxima
    static constexpr int XL_OFF = XM_OFF + 2 * 2 * kPM * 4;          // fp32 [half][128]: partial sums
    static constexpr int BAR_OFF = XL_OFF + 2 * kPM * 4;
    // barriers (arrivals per phase): raw_full[RS] (copy bytes), k_ready[2] (2 K warps),
    // v_ready[2] (4 V warps), s_full (commit), s_free[2] (8 softmax warps), p_ready (8),
    // pv_done[2] (commit), fin (2 commits), x[4 lane quarters] (the 2 warps of a quarter)
    static constexpr int B_RAW = 0, B_KR = RS, B_VR = RS + 2, B_SFULL = RS + 4, B_SFREE = RS + 5;
    static constexpr int B_PREADY = RS + 7, B_PV = RS + 8, B_FIN = RS + 10, B_X = RS + 11, NBAR = RS + 15;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;              // tmem base, bad flag
    static constexpr int SMEM = MISC_OFF + 16;
    static_assert(RAW % 16 == 0 && R_KS % 16 == 0 && R_V % 16 == 0 && R_VS % 16 == 0, "16-byte granules");
    static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
    static_assert(RAW_OFF < (1 << 18), "operand addresses must fit the descriptor's 18-bit field");
};

// ---- tcgen05 (5th-generation tensor core) helpers ----
// Shared-memory matrix descriptor: start address, leading (K-direction) and
// stride (row-group) byte offsets, all in 16-byte units; bits 46-48 hold the
// fixed value 0b001; base offset 0, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
           ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 D, fp16 A and B, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// D (+)= A.B, kind::f16, A in tensor memory (row r in lane r, two fp16 k
// elements per 32-bit column, k-step columns [a, a + 8)), B a shared-memory
// descriptor.  Issued by one elected lane of a converged warp whose lanes all
// pass the same (warp-uniform) operands: cheaper to issue than from inside a
// lane-0 branch, which has to take the uniform operands out of a divergent lane.
__device__ __forceinline__ void umma_f16_ta_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
                 " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
                 : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this
// warp's elected lane is done (elect.sync picks the same lane each time for
// the same full warp, so it is the lane that issued the MMAs).
__device__ __forceinline__ void umma_commit_w(uint32_t bar)
{
    asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
                 " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                 "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar) : "memory");
}

// Eight signed int8 codes (two words) -> eight exact fp16 values (16 bytes):
// the byte, biased by 128, goes under the binary16 exponent of 1024
// (0x64XX = 1024 + XX), and 1152 = 1024 + 128 is taken off.
__device__ __forceinline__ uint4 i8x8_to_f16(uint32_t w0, uint32_t w1)
{
    const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));
    const uint32_t x0 = w0 ^ 0x80808080u, x1 = w1 ^ 0x80808080u;
    uint32_t r[4] = {__byte_perm(x0, 0x64646464u, 0x4140), __byte_perm(x0, 0x64646464u, 0x4342),
                     __byte_perm(x1, 0x64646464u, 0x4140), __byte_perm(x1, 0x64646464u, 0x4342)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&r[k]), k1152);
        r[k] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// v = code * d2 (per position of the pair), as hi = fp16(v) and lo = fp16(v - hi)
// (the fused fp16 multiply-add rounds the exact v - hi once).
__device__ __forceinline__ void v_hilo(uint32_t code2, __half2 d2, uint32_t &hi, uint32_t &lo)
{
    const __half2 c = *reinterpret_cast<const __half2 *>(&code2);
    const __half2 h = __hmul2(c, d2);
    const __half2 l = __hfma2(c, d2, __hneg2(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <int VT, bool DUMP>
__global__ void __launch_bounds__(kPThreads, 1) prefill_attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = PrefillCfg<VT>;
    constexpr float kSlack = 3.0f;
    constexpr uint32_t kIdQK = umma_idesc_f16(kPM, kPN), kIdPV = umma_idesc_f16(kPM, kD);
    extern __shared__ __align__(1024) uint8_t smem[];

    // ---- the group, sequence, kv head, split and row tile of this CTA ----
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if ((int)blockIdx.x >= p.grp[k].cta0) gi = k;
    const GroupDesc &G = p.grp[gi];
    const int lb = (int)blockIdx.x - G.cta0;
    int rt, split, h, b;
    if (G.split_major) {   // every unit's split 0 first (the large pieces of an uneven split)
        const int per = G.n_rt * G.n_kv_heads * G.n_seqs, x = lb % per;
        split = lb / per;
        rt = x % G.n_rt;
        h = (x / G.n_rt) % G.n_kv_heads;
        b = x / G.n_rt / G.n_kv_heads;
    } else {
        const int ls = lb / G.n_rt;
        rt = lb % G.n_rt;
        split = ls % G.n_split;
        h = (ls / G.n_split) % G.n_kv_heads;
        b = ls / G.n_split / G.n_kv_heads;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gb = p.grp_begin[G.head0 + h], gsz = p.grp_begin[G.head0 + h + 1] - gb;
    const int row0 = rt * kPM;
    const int R = min(kPM, gsz * G.t_q - row0);
    if (R <= 0) return;   // a row tile past this kv head's rows (smaller group)
    const int seg0 = p.seq_seg0[G.seq0 + b], nseg = p.seq_nseg[G.seq0 + b];
    const int lcap = nseg ? min(G.max_len, p.seg[seg0 + nseg - 1].pos0 + p.seg[seg0 + nseg - 1].cap) : 0;

    pdl_wait();
    pdl_trigger();
    const int L = max(0, min(G.seq_lens[b], lcap));
    // the split's positions, cut at the sequence length and, under the causal
    // tail, after the last position the tile's last query token sees
    const int r0 = split == 0 ? 0 : G.chunk0 + (split - 1) * G.chunk;
    int r1 = min(L, split == 0 ? G.chunk0 : r0 + G.chunk);
    if (G.causal) r1 = min(r1, L - G.t_q + (row0 + R - 1) / gsz + 1);
    if (r0 >= r1) {   // nothing visible in this split
        if (!DUMP && tid < R) {
            const int i = (row0 + tid) / gsz, hq = p.grp_q[gb + (row0 + tid) % gsz];
            const size_t row = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
            if (G.n_split == 1) {
                G.lse[row] = -INFINITY;
                for (int d = 0; d < kD; ++d) G.out[row * kD + d] = 0.f;
            } else {
                G.ws_lse[row * G.n_split + split] = -INFINITY;
            }
        }
        return;
    }
    // KV tiles: each segment piece of [r0, r1) in runs of up to kPSub cache tiles
    int n_tiles = 0;
    for (int k = 0; k < nseg; ++k) {
        const SegDesc &s = p.seg[seg0 + k];
        const int end = (k + 1 < nseg) ? p.seg[seg0 + k + 1].pos0 : s.pos0 + s.cap;
        const int a = max(r0, s.pos0), e = min(min(r1, end), s.pos0 + s.cap);
        if (a < e) {
            const int n16 = (e - s.pos0 + kWTile - 1) / kWTile - (a - s.pos0) / kWTile;
            n_tiles += (n16 + kPSub - 1) / kPSub;
        }
    }

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::BAR_OFF;
    auto bar = [&](int k) { return bars + 8u * (uint32_t)k; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *bad = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    if (warp == kPCtlWarp) tmem_alloc(smem_u32(tmem_slot), 512);
    if (tid == 0) {
        *bad = 0;
        for (int k = 0; k < C::NBAR; ++k) {
            int n = kPSoftWarps;                                                        // s_free, p_ready
            if (k < C::RS || k == C::B_SFULL || k == C::B_PV || k == C::B_PV + 1) n = 1;
            else if (k == C::B_KR || k == C::B_KR + 1 || k == C::B_FIN || k >= C::B_X) n = 2;
            else if (k == C::B_VR || k == C::B_VR + 1) n = 4;
            mbar_init(bar(k), n);
        }
        fence_mbar_init();
    }

    // ---- softmax warps: warp w takes the 32 tile rows of its TMEM lane
    // quarter w%4 and, of each KV tile, positions 32(w/4)..+31; in the
    // prologue it quantizes blocks 2(w/4), 2(w/4)+1 of its row.  Rows are
    // numbered from lane quarter 2 on (rows 0-31 in lanes 64-95, 32-63 in
    // 96-127, then 0-31 and 32-63): a tile of up to 64 rows then runs its
    // softmax on SMSPs 2 and 3, beside the issuer warps, rather than on 0 and
    // 1, beside the K converters ----
    const bool srole = warp < kPSoftWarps;
    const int quarter = warp & 3, hf = (warp >> 2) & 1;
    const int rq = (quarter + 2) & 3;        // the quarter's place in the row order
    const int row = 32 * rq + lane;
    const bool row_ok = srole && row < R;
    int lim = -1;                            // last visible position of the row
    size_t orow = 0;
    tc_fence_before();
    __syncthreads();   // barriers and the TMEM base in place
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S_b at 64b (0..255), O at 256..383, the Q codes at 384..447
    // and P at 448..479 (high parts), 480..511 (low parts); fp16 A operands
    // hold two k elements per 32-bit column, row r in lane r
    const uint32_t tS = tmem, tO = tmem + 4 * kPN, tQ = tmem + 4 * kPN + kD, tPH = tQ + kD / 2, tPL = tPH + kPN / 2;
    if (srole) {   // Q codes of this row's two blocks -> TMEM columns 32hf.. of the Q area
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        float *qsl_s = reinterpret_cast<float *>(smem + C::QSL_OFF);
        const uint4 *src = nullptr;
        if (row_ok) {
            const int i = (row0 + row) / gsz, hq = p.grp_q[gb + (row0 + row) % gsz];
            orow = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
            lim = G.causal ? L - G.t_q + i : L - 1;
            src = reinterpret_cast<const uint4 *>(G.q + orow * kD);
        }
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
            const int bb = 2 * hf + b2;
            uint32_t wv[16];
            float sc = 0.f;
            if (row_ok) {
                float x[32];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 w = src[4 * bb + k];
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
                        x[8 * k + 2 * e] = f.x;
                        x[8 * k + 2 * e + 1] = f.y;
                    }
                }
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < 32; ++k) a = fmaxf(a, fabsf(x[k]));
                sc = __half2float(__float2half_rn(__fdiv_rn(a, 127.f)));
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    wv[e] = pack_half2((float)quant_i8(x[2 * e], sc), (float)quant_i8(x[2 * e + 1], sc));
                if (DUMP && split == 0) {   // the block's 32 codes and its scale bits
                    uint32_t cw[8];
#pragma unroll
                    for (int w4 = 0; w4 < 8; ++w4) {
                        cw[w4] = 0u;
#pragma unroll
                        for (int e = 0; e < 4; ++e) cw[w4] |= (uint32_t)(quant_i8(x[4 * w4 + e], sc) & 0xff) << (8 * e);
                    }
                    uint4 *qd = reinterpret_cast<uint4 *>(G.dbg_qc + orow * kD + 32 * bb);
                    qd[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    qd[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                    G.dbg_qs[orow * kNB + bb] = __half_as_ushort(__float2half_rn(sc));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) wv[e] = 0u;
            }
            qsl_s[row * kNB + bb] = sc * G.qk_scale_log2;
            tmem_st16(tQ + lane_base + 16 * bb, wv);   // dims 32bb.. -> columns 16bb..
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();   // the Q operand and the query scales in place
    tc_fence_after();

    // called by whole warps (a uniform decision): counted once per warp
    auto give_up = [&]() {
        if (lane == 0 && !*bad) {
            *bad = 1;
            atomicAdd(p.timeouts, 1u);
        }
    };
    // Warp-uniform wait.  Every wait of this kernel suspends the warp
    // (try_wait) rather than spinning on test_wait: four roles share each
    // SMSP, and a spinning waiter takes issue slots from the softmax warps
    // beside it (measured: the attention call 723 -> 711 us with the issuers'
    // and the softmax's waits suspending instead of spinning).
    auto wwait = [&](uint32_t b_, uint32_t parity) {
        const bool okw = mbar_wait(b_, parity);
        return __all_sync(0xffffffffu, okw);
    };
    auto wbad = [&]() { return __any_sync(0xffffffffu, *bad != 0); };

    if (warp == kPCtlWarp) {
        // ================= QK MMAs (the warp runs the loop, one elected lane
        // issues) =================
        // descriptors of the k16 steps differ from a base only in the start
        // address (16-byte units, no carry out of its 14 bits)
        const uint64_t dK0 = umma_desc(sbase + C::K_OFF, C::K_LBO, C::K_SBO);
        const uint64_t dK1 = umma_desc(sbase + C::K_OFF + C::KBUF, C::K_LBO, C::K_SBO);
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            if (!wwait(bar(C::B_KR + (j & 1)), (j >> 1) & 1)) { give_up(); break; }
            if (j > 0 && !wwait(bar(C::B_SFREE + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { give_up(); break; }
            tc_fence_after();
            const uint64_t dK = (j & 1) ? dK1 : dK0;
#pragma unroll
            for (int bb = 0; bb < kNB; ++bb)
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t o = (uint64_t)((4 * bb + 2 * kk) * (C::K_LBO / 16));
                    umma_f16_ta_w(tS + kPN * bb, tQ + 16 * bb + 8 * kk, dK + o, kIdQK, kk);
                }
            umma_commit_w(bar(C::B_SFULL));
        }
        umma_commit_w(bar(C::B_FIN));
        if (!wwait(bar(C::B_FIN), 0)) give_up();
    } else if (warp == kPPvWarp) {
        // ================= P.V MMAs as soon as each tile's P and V are in
        // place; the bulk copies of the tiles RS ahead (the warp runs the
        // loop, one elected lane issues) =================
        int4 *rec = reinterpret_cast<int4 *>(smem + C::REC_OFF);
        int *nsub = reinterpret_cast<int *>(smem + C::NSUB_OFF);
        Walk w;
        walk_seek(p, seg0, nseg, h, r0, r1, 0, C::VCODE, w);
        int issued = 0;
        auto issue = [&]() {
            const int st = issued % C::RS;
            const int n = min(kPSub, w.Tend - w.T);
            if (lane == 0) {
                for (int k = 0; k < kPSub; ++k) {
                    const int tb = (w.T + k) * kWTile;
                    rec[st * kPSub + k] = make_int4(tb, w.la, w.le, w.pos0 + tb);
                }
                nsub[st] = n;
            }
            __syncwarp();   // the records before the (elected lane's) arrival that publishes them
            const uint32_t dst = sbase + C::RAW_OFF + st * C::RAW, bw = bar(C::B_RAW + st);
            mbar_arrive_expect_tx_w(bw, n * C::TILE);
            bulk_g2s_w(dst + C::R_K, w.gk, n * C::TILE_K, bw);
            bulk_g2s_w(dst + C::R_KS, w.gks, n * C::TILE_S, bw);
            bulk_g2s_w(dst + C::R_V, w.gv, n * C::TILE_V, bw);
            bulk_g2s_w(dst + C::R_VS, w.gvs, n * C::TILE_S, bw);
            w.T += n;
            w.gk += n * C::TILE_K;
            w.gks += n * C::TILE_S;
            w.gv += n * C::TILE_V;
            w.gvs += n * C::TILE_S;
            if (w.T >= w.Tend) walk_seek(p, seg0, nseg, h, r0, r1, w.k + 1, C::VCODE, w);
            ++issued;
        };
        while (issued < min(C::RS, n_tiles)) issue();
        const uint64_t dVH0 = umma_desc(sbase + C::VH_OFF, 128, C::V_SBO);
        const uint64_t dVH1 = umma_desc(sbase + C::VH_OFF + C::VBUF, 128, C::V_SBO);
        const uint64_t dVL0 = umma_desc(sbase + C::VL_OFF, 128, C::V_SBO);
        const uint64_t dVL1 = umma_desc(sbase + C::VL_OFF + C::VBUF, 128, C::V_SBO);
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            if (!wwait(bar(C::B_PREADY), j & 1) || !wwait(bar(C::B_VR + (j & 1)), (j >> 1) & 1)) {
                give_up();
                break;
            }
            tc_fence_after();
            const uint64_t dVH = (j & 1) ? dVH1 : dVH0, dVL = (j & 1) ? dVL1 : dVL0;
#pragma unroll
            for (int ks = 0; ks < kPN / 16; ++ks) {
                const uint64_t o = (uint64_t)(16 * ks);   // 2 ks * 128 bytes
                umma_f16_ta_w(tO, tPH + 8 * ks, dVH + o, kIdPV, (j > 0 || ks > 0) ? 1u : 0u);
                umma_f16_ta_w(tO, tPL + 8 * ks, dVH + o, kIdPV, 1u);
                umma_f16_ta_w(tO, tPH + 8 * ks, dVL + o, kIdPV, 1u);
            }
            umma_commit_w(bar(C::B_PV + (j & 1)));
            // both converters are done with tile j's stage (the V warps
            // said so; the K warps before the softmax passed tile j)
            if (issued < n_tiles) issue();
        }
        // drain: every MMA issued here, and the copies no converter took
        umma_commit_w(bar(C::B_FIN));
        if (!wwait(bar(C::B_FIN), 0)) give_up();
        for (int k = max(0, issued - C::RS); k < issued; ++k) mbar_wait(bar(C::B_RAW + k % C::RS), (k / C::RS) & 1);
    } else if (warp >= kPKWarp0) {
        // ================= convert: cache codes -> fp16 operands =================
        // K warps: K codes, K scales, the slot records (K(j) may overwrite
        // tile j-2's once the softmax has read S(j-2)).  V warps: V hi / lo
        // (once P.V(j-2) is done).
        const bool kside = warp < kPVWarp0;
        const int kw = warp - kPKWarp0, ct = tid - 32 * kPVWarp0;
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            const int st = j % C::RS, ob = j & 1;
            if (!wwait(bar(C::B_RAW + st), (j / C::RS) & 1)) { give_up(); break; }
            if (j >= 2 && !wwait(kside ? bar(C::B_SFREE + ob) : bar(C::B_PV + ob), ((j - 2) >> 1) & 1)) {
                give_up();
                break;
            }
            const uint8_t *raw = smem + C::RAW_OFF + st * C::RAW;
            const int4 *rec = reinterpret_cast<const int4 *>(smem + C::REC_OFF) + st * kPSub;
            const int ns = reinterpret_cast<const int *>(smem + C::NSUB_OFF)[st];
            // slot k (sub-tile k / 16, position k % 16) holds a visible cache
            // row?  One bit per slot, from two ballots of the warp.
            uint64_t vmask;
            {
                bool v2[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int k = 32 * hh + lane, t4 = k / kWTile, u = k % kWTile;
                    const int4 r = rec[t4];
                    v2[hh] = t4 < ns && r.x + u >= r.y && r.x + u < r.z && r.w + u < L;
                }
                vmask = (uint64_t)__ballot_sync(0xffffffffu, v2[0]) | ((uint64_t)__ballot_sync(0xffffffffu, v2[1]) << 32);
            }
            auto slot_ok = [&](int t4, int u) { return (vmask >> (kWTile * t4 + u)) & 1ull; };
            if (kside) {
            const int kt = 32 * kw + lane;   // 0..63
            if (kt < kPSub) reinterpret_cast<int4 *>(smem + C::OREC_OFF)[ob * kPSub + kt] = rec[kt];
            if (kt == 0) reinterpret_cast<int *>(smem + C::ONSUB_OFF)[ob] = ns;
            // K codes: 16-byte chunk i of a cache tile (i = 2kw, 2kw + 1 here)
            // holds position 8(i/2) + lane/4, dims 64(i%2) + 8(lane%4) + 0..7
            // and the same + 32
            uint8_t *kop = smem + C::K_OFF + ob * C::KBUF;
#pragma unroll
            for (int t4 = 0; t4 < kPSub; ++t4)
#pragma unroll
                for (int ii = 0; ii < 2; ++ii) {
                    const int i = 2 * kw + ii;
                    const int u = 8 * (i >> 1) + (lane >> 2), pos = kWTile * t4 + u;
                    const int dg0 = 8 * (i & 1) + (lane & 3);
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                    if (slot_ok(t4, u)) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(raw + C::R_K + t4 * C::TILE_K + i * 512 + lane * 16);
                        lo = i8x8_to_f16(w.x, w.y);
                        hi = i8x8_to_f16(w.z, w.w);
                    }
                    *reinterpret_cast<uint4 *>(kop + (pos / 8) * C::K_SBO + dg0 * C::K_LBO + (pos % 8) * 16) = lo;
                    *reinterpret_cast<uint4 *>(kop + (pos / 8) * C::K_SBO + (dg0 + 4) * C::K_LBO + (pos % 8) * 16) = hi;
                }
            // K scales as fp32 [block][position]
            {
                const int ct = kt;
                const int t4 = ct / kWTile, u = ct % kWTile;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (slot_ok(t4, u)) {
                    float x[4];
                    load4h(reinterpret_cast<const uint16_t *>(raw + C::R_KS + t4 * C::TILE_S) + u * kNB, x);
                    v = make_float4(x[0], x[1], x[2], x[3]);
                }
                float *skf = reinterpret_cast<float *>(smem + C::SKF_OFF) + ob * kNB * kPN;
                skf[0 * kPN + ct] = v.x;
                skf[1 * kPN + ct] = v.y;
                skf[2 * kPN + ct] = v.z;
                skf[3 * kPN + ct] = v.w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_KR + ob));
            } else {
            // V: v / 2 = code * (d / 2) as fp16 hi + lo, stored [dim][position]
            uint8_t *vh = smem + C::VH_OFF + ob * C::VBUF, *vl = smem + C::VL_OFF + ob * C::VBUF;
            auto put = [&](int dim, int pos, uint32_t code2, __half2 d2) {
                uint32_t hi, lo;
                v_hilo(code2, d2, hi, lo);
                const int o = (dim / 8) * C::V_SBO + (pos / 8) * 128 + (dim % 8) * 16 + (pos % 8) * 2;
                *reinterpret_cast<uint32_t *>(vh + o) = hi;
                *reinterpret_cast<uint32_t *>(vl + o) = lo;
            };
            constexpr int NCH = kPSub * C::TILE_V / 16 / 128;   // 16-byte chunks per converter thread
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
                const int cidx = ct + 128 * k;                   // chunk of the KV tile
                const int t4 = cidx / (C::TILE_V / 16), ci = cidx % (C::TILE_V / 16);
                const int i = ci / 32, ln = ci % 32, g = ln >> 2, c = ln & 3;
                const uint4 w = *reinterpret_cast<const uint4 *>(raw + C::R_V + t4 * C::TILE_V + ci * 16);
                const int t = (VT == KVQ_V_Q4_0) ? 8 * i + 2 * c : 8 * (i >> 1) + 2 * c;
                const int pos = kWTile * t4 + t;
                // scales of positions t, t + 1 (0 where the slot holds no visible row), times 1/2
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                const uint16_t *vs = reinterpret_cast<const uint16_t *>(raw + C::R_VS + t4 * C::TILE_S);
                if (slot_ok(t4, t)) load4h(vs + t * kNB, d0);
                if (slot_ok(t4, t + 1)) load4h(vs + (t + 1) * kNB, d1);
                if (VT == KVQ_V_Q4_0) {
                    const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));   // 1032
                    const __half2 k16th = __half2half2(__ushort_as_half(0x2c00));   // 1/16
                    const __half2 km72 = __half2half2(__ushort_as_half(0xd480));    // -72
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int bb = 0; bb < kNB; ++bb) {
                        const __half2 d2 = __floats2half2_rn(d0[bb] * kPVScale, d1[bb] * kPVScale);
                        const uint32_t w0 = ws[bb], w23 = w0 >> 8;
                        uint32_t x;
                        __half2 cv;
                        x = (w0 & 0x000F000Fu) | 0x64006400u;
                        cv = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
                        put(32 * bb + 2 * g, pos, *reinterpret_cast<uint32_t *>(&cv), d2);
                        x = (w23 & 0x000F000Fu) | 0x64006400u;
                        cv = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
                        put(32 * bb + 2 * g + 1, pos, *reinterpret_cast<uint32_t *>(&cv), d2);
                        x = (w0 & 0x00F000F0u) | 0x64006400u;
                        cv = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
                        put(32 * bb + 2 * g + 16, pos, *reinterpret_cast<uint32_t *>(&cv), d2);
                        x = (w23 & 0x00F000F0u) | 0x64006400u;
                        cv = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
                        put(32 * bb + 2 * g + 17, pos, *reinterpret_cast<uint32_t *>(&cv), d2);
                    }
                } else {
                    const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));   // 1152
                    const int hb = i & 1;
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int bb = 2 * hb + half;
                        const float e0 = hb ? d0[2 + half] : d0[half], e1 = hb ? d1[2 + half] : d1[half];
                        const __half2 d2 = __floats2half2_rn(e0 * kPVScale, e1 * kPVScale);
#pragma unroll
                        for (int wd = 0; wd < 2; ++wd) {
                            const uint32_t xw = ws[2 * half + wd] ^ 0x80808080u;
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                uint32_t x = __byte_perm(xw, 0x64646464u, e ? 0x4342 : 0x4140);
                                const __half2 cv = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
                                put(32 * bb + 4 * g + 2 * wd + e, pos, *reinterpret_cast<const uint32_t *>(&cv), d2);
                            }
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_VR + ob));
            }
        }
    } else {
        // ================= softmax: scores, P, final O =================
        // This thread: tile row `row` (TMEM lane), positions 32hf..32hf+31 of
        // each KV tile, head-dim columns 64hf..64hf+63 of O.  The two halves of
        // a row agree on its reference max through the tile-max exchange, and
        // keep their own partial sums l.
        if (32 * rq >= R) {
            // No query row in this TMEM lane quarter (a tile of up to 32 rows,
            // or the ragged last one): keep the barrier phases in step with
            // the live warps and do nothing else.  Per tile: S(j) complete,
            // the two arrivals the issuers count (S read, P written; the rows
            // here feed nothing the output keeps), then the P-ready phase's
            // completion, so that no arrival for tile j + 1 lands in phase j.
            for (int j = 0; j < n_tiles; ++j) {
                if (wbad()) break;
                if (!wwait(bar(C::B_SFULL), j & 1)) { give_up(); break; }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(C::B_SFREE + (j & 1)));
                    mbar_arrive(bar(C::B_PREADY));
                }
                if (!wwait(bar(C::B_PREADY), j & 1)) { give_up(); break; }
            }
        } else {
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        float qsl[kNB];   // block scale * sm_scale * log2(e)
        {
            const float4 q4 = reinterpret_cast<const float4 *>(smem + C::QSL_OFF)[row];
            qsl[0] = q4.x; qsl[1] = q4.y; qsl[2] = q4.z; qsl[3] = q4.w;
        }
        float *xm = reinterpret_cast<float *>(smem + C::XM_OFF);   // [parity][half][row]
        float m = -INFINITY, l = 0.f, mu = 0.f;
        bool o_live = false;   // O holds an earlier tile's P.V
        constexpr int HP = kPN / 2;   // positions per half
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            const int ob = j & 1;
            // this tile's scores, and (directly from the converters) its K
            // scales and slot records
            if (!wwait(bar(C::B_SFULL), j & 1) || !wwait(bar(C::B_KR + ob), (j >> 1) & 1)) { give_up(); break; }
            tc_fence_after();
            const float *skf = reinterpret_cast<const float *>(smem + C::SKF_OFF) + ob * kNB * kPN + HP * hf;
            float s[HP];
#pragma unroll
            for (int q = 0; q < HP / 16; ++q) {
                uint32_t a[kNB][16];
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) tmem_ld16(tS + lane_base + kPN * bb + HP * hf + 16 * q, a[bb]);
                tmem_wait_ld();
                if constexpr (DUMP) {
                    // positions 16 q + u of this half: sub-tile 2 hf + q of the KV tile
                    const int4 r = reinterpret_cast<const int4 *>(smem + C::OREC_OFF)[ob * kPSub + 2 * hf + q];
                    const int nsd = reinterpret_cast<const int *>(smem + C::ONSUB_OFF)[ob];
                    if (row_ok && 2 * hf + q < nsd) {
#pragma unroll
                        for (int u = 0; u < kWTile; ++u) {
                            const int tok = r.x + u, pos = r.w + u;
                            if (tok >= r.y && tok < r.z && pos < L)
                                *reinterpret_cast<int4 *>(G.dbg_scores + (orow * G.max_len + pos) * kNB) =
                                    make_int4((int)__uint_as_float(a[0][u]), (int)__uint_as_float(a[1][u]),
                                              (int)__uint_as_float(a[2][u]), (int)__uint_as_float(a[3][u]));
                        }
                    }
                }
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4) {
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0;
#pragma unroll
                    for (int bb = 0; bb < kNB; ++bb) {
                        const float4 k4 = *reinterpret_cast<const float4 *>(skf + bb * kPN + 16 * q + jj);
                        const float2 qq = make_float2(qsl[bb], qsl[bb]);
                        acc0 = fma2(mul2(make_float2(__uint_as_float(a[bb][jj]), __uint_as_float(a[bb][jj + 1])), qq),
                                    make_float2(k4.x, k4.y), acc0);
                        acc1 = fma2(mul2(make_float2(__uint_as_float(a[bb][jj + 2]), __uint_as_float(a[bb][jj + 3])), qq),
                                    make_float2(k4.z, k4.w), acc1);
                    }
                    s[16 * q + jj] = acc0.x;
                    s[16 * q + jj + 1] = acc0.y;
                    s[16 * q + jj + 2] = acc1.x;
                    s[16 * q + jj + 3] = acc1.y;
                }
            }
            // mask slots without a visible cache row or past the row's limit
            // (this half holds sub-tiles 2hf, 2hf + 1)
            const int4 *rec = reinterpret_cast<const int4 *>(smem + C::OREC_OFF) + ob * kPSub;
            const int ns = reinterpret_cast<const int *>(smem + C::ONSUB_OFF)[ob];
            const int lim_r = min(lim, L - 1);
            bool full = true;
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {
                const int t4 = 2 * hf + t2;
                const int4 r = rec[t4];
                full = full && t4 < ns && r.x >= r.y && r.x + kWTile <= r.z && r.w + kWTile - 1 <= lim_r;
            }
            if (!full) {
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2) {
                    const int t4 = 2 * hf + t2;
                    const int4 r = rec[t4];
                    const bool live = t4 < ns;
#pragma unroll
                    for (int u = 0; u < kWTile; ++u) {
                        const int tok = r.x + u, pos = r.w + u;
                        const bool ok = live && tok >= r.y && tok < r.z && pos <= lim_r;
                        s[kWTile * t2 + u] = ok ? s[kWTile * t2 + u] : -INFINITY;
                    }
                }
            }
            // S(j), the K scales and the slot records of tile j are read: the
            // next QK and the K converters may go on
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_SFREE + ob));
            // tile max of this half: four running maxima, then a tree (a
            // dependency chain of 10 instead of 31)
            float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
            for (int k = 4; k < HP; k += 4)
#pragma unroll
                for (int e = 0; e < 4; ++e) m4[e] = fmaxf(m4[e], s[k + e]);
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            // the row's tile max over both halves
            xm[(ob * 2 + hf) * kPM + row] = mx;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_X + quarter));
            if (!wwait(bar(C::B_X + quarter), j & 1)) { give_up(); break; }
            mx = fmaxf(mx, xm[(ob * 2 + (hf ^ 1)) * kPM + row]);
            const bool need = mx > m + kSlack;
            const bool wneed = o_live && __any_sync(0xffffffffu, need);   // rescale O (whole warp)
            float alpha = 1.f;
            if (need) {
                const float mnew = fmaxf(m, mx);
                alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - mnew);
                l *= alpha;
                m = mnew;
                mu = m;
            }
            float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // two running pair sums
#pragma unroll
            for (int k = 0; k < HP; k += 2) {
                const float2 t = sub2(make_float2(s[k], s[k + 1]), make_float2(mu, mu));
                s[k] = fast_exp2(t.x);
                s[k + 1] = fast_exp2(t.y);
                ls2[(k >> 1) & 1] = add2(ls2[(k >> 1) & 1], make_float2(s[k], s[k + 1]));
            }
            const float2 lsum = add2(ls2[0], ls2[1]);
            l += lsum.x + lsum.y;
            // P(j) may overwrite P(j-1) once P.V(j-1) is done; O is then stable
            if (j > 0) {
                if (!wwait(bar(C::B_PV + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { give_up(); break; }
                tc_fence_after();
            }
            if (wneed) {   // O *= alpha on this half's columns (1 on the rows that keep their max)
#pragma unroll
                for (int c0 = 0; c0 < kD / 2; c0 += 16) {
                    uint32_t o[16];
                    tmem_ld16(tO + lane_base + (kD / 2) * hf + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                    tmem_st16(tO + lane_base + (kD / 2) * hf + c0, o);
                }
                tmem_wait_st();
            }
            {   // P of this half: positions 32hf.. -> columns 16hf.. of the P areas
                uint32_t hw[HP / 2], lw[HP / 2];
#pragma unroll
                for (int e = 0; e < HP / 2; ++e) {
                    const float2 x = make_float2(s[2 * e], s[2 * e + 1]);
                    const uint32_t hp = pack_half2(x.x, x.y);
                    const float2 hf2 = __half22float2(*reinterpret_cast<const __half2 *>(&hp));
                    const float2 lo = sub2(x, hf2);
                    hw[e] = hp;
                    lw[e] = pack_half2(lo.x, lo.y);
                }
                tmem_st16(tPH + lane_base + (HP / 2) * hf, hw);
                tmem_st16(tPL + lane_base + (HP / 2) * hf, lw);
                tmem_wait_st();
            }
            o_live = true;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PREADY));
        }
        // ---- final O of this row: the halves' partial sums, then each half
        // writes its 64 columns ----
        bool ok = !wbad() && n_tiles > 0;
        float *xl = reinterpret_cast<float *>(smem + C::XL_OFF);
        if (ok) {
            ok = wwait(bar(C::B_PV + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1);
            tc_fence_after();
            if (ok) {
                xl[hf * kPM + row] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_X + quarter));
                ok = wwait(bar(C::B_X + quarter), n_tiles & 1);
            }
            if (!ok) give_up();
        }
        const bool lost = !ok || wbad();
        if (DUMP) {
            // the test hook writes no out / lse
        } else if (lost) {   // results lost: NaN rows
            if (row_ok) {
                const float nan = __int_as_float(0x7fc00000);
                if (G.n_split == 1) {
                    if (hf == 0) G.lse[orow] = nan;
                    for (int d = 0; d < kD / 2; ++d) G.out[orow * kD + (kD / 2) * hf + d] = nan;
                } else {
                    if (hf == 0) G.ws_lse[orow * G.n_split + split] = nan;
                    for (int d = 0; d < kD / 2; ++d) G.ws_o[(orow * G.n_split + split) * kD + (kD / 2) * hf + d] = nan;
                }
            }
        } else {
            const float lt = l + xl[(hf ^ 1) * kPM + row];
            const bool any = lt > 0.f;
            float inv, lg;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(lt));
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(lt));
            const float f = any ? inv / kPVScale : 0.f;
            const float lse = any ? (m + lg) * 0.69314718055994531f : -INFINITY;
            float *dst = ((G.n_split == 1) ? G.out + orow * kD : G.ws_o + (orow * G.n_split + split) * kD) + (kD / 2) * hf;
#pragma unroll
            for (int c0 = 0; c0 < kD / 2; c0 += 16) {
                uint32_t o[16];
                tmem_ld16(tO + lane_base + (kD / 2) * hf + c0, o);   // every lane of the warp takes part
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int k = 0; k < 16; k += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + k) =
                            make_float4(any ? __uint_as_float(o[k]) * f : 0.f, any ? __uint_as_float(o[k + 1]) * f : 0.f,
                                        any ? __uint_as_float(o[k + 2]) * f : 0.f, any ? __uint_as_float(o[k + 3]) * f : 0.f);
                }
            }
            if (row_ok && hf == 0) {
                if (G.n_split == 1) G.lse[orow] = lse;
                else G.ws_lse[orow * G.n_split + split] = lse;
            }
        }
        }   // live quarter
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPCtlWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int VT>
cudaError_t launch_prefill_t(const AttnParams &p, int n_ctas, bool dump, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = PrefillCfg<VT>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (dump) return cudaLaunchKernelEx(&cfg, prefill_attn_kernel<VT, true>, p);
    return cudaLaunchKernelEx(&cfg, prefill_attn_kernel<VT, false>, p);
}

template <int VT>
cudaError_t prepare_prefill_t()
{
    const cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel<VT, false>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, PrefillCfg<VT>::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(prefill_attn_kernel<VT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PrefillCfg<VT>::SMEM);
}

}  // namespace kvq
