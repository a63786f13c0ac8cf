// kvq_attn.cuh -- split-KV decode attention over the quantized cache (sm_103a).
//
// One CTA = (row tile, split s, kv head h, sequence b) of one work group of the
// launch: it attends up to 8 NT query rows of kv head h (of its t_q query tokens
// x the query heads mapped to h) over the positions [s*chunk, (s+1)*chunk) of
// sequence b and writes either the final output (one split) or a partial
// (normalised o, lse) for the combine.
//
// Data path: every warp streams its own contiguous share of the CTA's
// positions through a private ring of 16-position stages in shared memory.
// The cache stores each 16-position tile of every array contiguously, with the
// code bytes already in the order the MMA fragments read them (the tile layout
// in kvq_internal.cuh), so one lane fills a stage with four bulk async copies
// (cp.async.bulk, completion counted in bytes on the stage's mbarrier) and
// every fragment read is one conflict-free 16-byte shared load.  Only
// __syncwarp and the stage barriers run in the main loop; the block
// synchronizes once for the query prologue and once to merge the warps.
//
//   * QK^T: fp16 tensor-core MMA m16n8k16 on exact integers -- A = the K codes
//     of the stage's 16 positions entered as 1152 + code (one xor and two
//     byte-permutes per packed word), B = 8 query rows' codes, two MMAs per
//     32-block into one accumulator that starts at -1152 * (sum of the row's
//     codes in the block).  Every partial sum is an integer below 2^24, so the
//     fp32 accumulator ends exactly at the integer block dot I_b (never summed
//     across blocks before scaling).  (GB300's int8 mma.sync issues ~8x slower
//     than the fp16 one, which is why the integer dot runs on the fp16 path.)
//     Each lane ends up with positions g, g + 8 of rows 2c, 2c + 1.
//   * score = sum_b I_b * (sq_b * sk_b) * sm_scale*log2(e), masked to -inf
//     outside the sequence / causal range; online softmax in base 2 with the
//     row's reference max only raised when a score passes it by more than 3
//     (p <= 8), which skips the cross-lane max on almost every stage.
//   * P.V: fp16 tensor-core MMA m16n8k16 with fp32 accumulation.  The V codes
//     enter as exact small integers in fp16 (binary16 exponent trick: 0x6400|n
//     is 1024+n).  The tile layout puts the same head dims of two adjacent
//     positions side by side, which gives the (position, position) pairs the
//     MMA's k dimension needs without a transpose.  The per-(position, block)
//     scale d rides on the P side: B = p*d split into an fp16 high part and an fp16 low part (two MMAs), so
//     P.V keeps ~22 bits of the fp32 product; each part is packed at
//     (position, row) and turned to (row, position) order with movmatrix.  The
//     P.V accumulators' columns are the same rows 2c, 2c + 1, so the softmax
//     rescale needs no shuffles.
//
// Each warp keeps its own (m, l, acc); the warps' states are merged through
// shared memory at the end in a fixed order.
#pragma once

#include <type_traits>

#include "kvq_internal.cuh"

namespace kvq {

#ifndef KVQ_STAGES_Q4
#define KVQ_STAGES_Q4 2   // stages per warp ring (q4_0 V)
#endif
#ifndef KVQ_TPS_Q4
#define KVQ_TPS_Q4 2      // 16-position tiles per stage (q4_0 V)
#endif
#ifndef KVQ_STAGES_Q8
#define KVQ_STAGES_Q8 3   // (q8_0 V)
#endif
#ifndef KVQ_TPS_Q8
#define KVQ_TPS_Q8 1
#endif



template <int NT, int VT, int KT = KVQ_K_I8, int W = split_warps(NT)>
struct SplitCfg {
    static constexpr int WARPS = W;
    static constexpr int THREADS = WARPS * 32;
    // the <= 8-row kernels are held to 128 registers per thread (512 threads per SM x 4 CTAs of 4 warps,
    // or one CTA of 16 warps); the others take what they need
    static constexpr int MIN_CTAS = (NT == 1) ? (16 / WARPS > 0 ? 16 / WARPS : 1) : 1;
    static constexpr int QROWS = (8 * NT > WARPS) ? 8 * NT : WARPS;   // query rows kept in smem
    static_assert(QROWS % WARPS == 0, "every warp quantizes the same number of query rows");
    static constexpr bool F16K = KT == KVQ_K_F16;
    // ring depth per warp and tiles per stage (F16 K tiles are twice as large)
    static constexpr int STAGES = F16K ? 2 : (VT == KVQ_V_Q4_0) ? KVQ_STAGES_Q4 : KVQ_STAGES_Q8;
    static constexpr int TPS = F16K ? 1 : (VT == KVQ_V_Q4_0) ? KVQ_TPS_Q4 : KVQ_TPS_Q8;
    static constexpr int VCODE = (VT == KVQ_V_Q4_0) ? kD / 2 : kD;            // V code bytes per position
    static constexpr int KCODE = F16K ? 2 * kD : kD;                          // K bytes per position
    static constexpr int TILE_K = kWTile * KCODE, TILE_S = kWTile * kNB * 2, TILE_V = kWTile * VCODE;
    static constexpr int TILE_KS = F16K ? 0 : TILE_S;                         // K scales (none for F16 K)
    static constexpr int TILE = TILE_K + TILE_KS + TILE_V + TILE_S;           // bytes of one tile
    // one warp stage: up to TPS consecutive tiles of one segment, each array's
    // tiles side by side as in the cache (K codes, K scales, V codes, V scales)
    static constexpr int K_OFF = 0;
    static constexpr int KS_OFF = K_OFF + TPS * TILE_K;
    static constexpr int V_OFF = KS_OFF + TPS * TILE_KS;
    static constexpr int VS_OFF = V_OFF + TPS * TILE_V;
    static constexpr int STAGE = VS_OFF + TPS * TILE_S;
    static constexpr int RING = STAGES * STAGE;               // per warp
    // The query rows' codes, scales and code sums are read only while the
    // query table below is built.  Every warp hands its first STAGES - 1 ring
    // slots to the copy engine before that and its last slot only in the main
    // loop, so they sit in the last warp's last slot when they fit there.
    static constexpr int QBYTES = QROWS * KCODE + 2 * QROWS * kNB * 4;
    static constexpr bool Q_IN_RING = QBYTES <= STAGE;
    static constexpr int Q_OFF = Q_IN_RING ? (WARPS - 1) * RING + (STAGES - 1) * STAGE : WARPS * RING;
    static constexpr int QS_OFF = Q_OFF + QROWS * KCODE;      // fp32 [QROWS][kNB]
    static constexpr int QSUM_OFF = QS_OFF + QROWS * kNB * 4; // int32 [QROWS][kNB]
    // Per-lane query table, [chunk][lane][4 words] (16-byte chunks, lane-major
    // so a warp's LDS.128 of one chunk is conflict free): per (8-row tile nt,
    // block) the query MMA B fragments of both k16 steps and the accumulator
    // seeds of the lane's two rows, and per (nt, row) the row's block scales.
    static constexpr int QB_CHUNKS = NT * kNB;
    static constexpr int SEED_CHUNKS = NT * kNB;
    static constexpr int SQ_CHUNKS = NT * 2;
    static constexpr int QF_CHUNKS = QB_CHUNKS + SEED_CHUNKS + SQ_CHUNKS;
    static constexpr int QF_OFF = Q_IN_RING ? WARPS * RING : (QSUM_OFF + QROWS * kNB * 4 + 15) / 16 * 16;
    static constexpr int OROW = kD + 4;                        // merge slice row (floats, padded)
    // The merge reuses the stage rings once every stage is consumed: one
    // [8*NT][OROW] slice per warp when they all fit (else one shared slice),
    // then m, l [WARPS][8*NT] and M, 1/L, lse [8*NT].
    static constexpr bool SLICES = WARPS * 8 * NT * OROW * 4 <= WARPS * STAGES * STAGE;
    static constexpr int ML_OFF = (SLICES ? WARPS : 1) * 8 * NT * OROW * 4;
    static constexpr int TI_OFF = QF_OFF + QF_CHUNKS * 32 * 16;  // int4 record of a stage's first tile [WARPS][STAGES]
    static constexpr int NS_OFF = TI_OFF + WARPS * STAGES * 16;         // int tiles in stage [WARPS][STAGES]
    static constexpr int NEW_OFF = (NS_OFF + WARPS * STAGES * 4 + 15) / 16 * 16;  // appended rows [KVQ_MAX_T_Q_APPEND][32 lanes][3 words]
    static constexpr int BAR_OFF = NEW_OFF + KVQ_MAX_T_Q_APPEND * 32 * 12;          // uint64 mbarrier [WARPS][STAGES]
    static constexpr int FLAG_OFF = BAR_OFF + WARPS * STAGES * 8;
    static constexpr int SMEM = FLAG_OFF + 16;
    static_assert(ML_OFF + (2 * WARPS + 3) * 8 * NT * 4 <= WARPS * RING, "merge buffers must fit in the stage rings");
    static_assert(STAGE % 16 == 0 && KS_OFF % 16 == 0 && V_OFF % 16 == 0 && VS_OFF % 16 == 0, "16-byte granules");
    static_assert(TPS == 1 || TPS == 2, "one or two tiles per stage");
    static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
};

// The warp (converged; one elected lane issues) fills ring slot `dst`
// (shared address) with n consecutive tiles of one segment starting at the
// walk's next tile: four contiguous bulk copies whose bytes complete on the
// slot's barrier.  Positions of a tile outside [la, le) are copied too (they
// are cache rows of the same segment, possibly never written) and masked where
// they are used.
template <int NT, int VT, int KT>
__device__ __forceinline__ void tile_issue(const Walk &w, int n, uint32_t dst, uint32_t bar)
{
    using C = SplitCfg<NT, VT, KT>;
    mbar_arrive_expect_tx_w(bar, n * C::TILE);
    bulk_g2s_w(dst + C::K_OFF, w.gk, n * C::TILE_K, bar);
    if (C::TILE_KS) bulk_g2s_w(dst + C::KS_OFF, w.gks, n * C::TILE_KS, bar);
    bulk_g2s_w(dst + C::V_OFF, w.gv, n * C::TILE_V, bar);
    bulk_g2s_w(dst + C::VS_OFF, w.gvs, n * C::TILE_S, bar);
}

// The same for a KVQ_LAYOUT_ROWS segment: only the rows [ra, rb) of the n
// tiles (relative to the first tile's token 0) that the piece covers, at their
// places in the slot; scale rows are copied in pairs (16-byte granules).  The
// other rows of the slot keep stale bytes, which the masks never let through.
template <int NT, int VT, int KT>
__device__ __forceinline__ void rows_issue(const Walk &w, int ra, int rb, uint32_t dst, uint32_t bar)
{
    using C = SplitCfg<NT, VT, KT>;
    const int sa = ra & ~1, sb = (rb + 1) & ~1;
    mbar_arrive_expect_tx_w(bar, (rb - ra) * (C::KCODE + C::VCODE) + (sb - sa) * 2 * kNB * 2);
    bulk_g2s_w(dst + C::K_OFF + ra * C::KCODE, w.gk + ra * C::KCODE, (rb - ra) * C::KCODE, bar);
    bulk_g2s_w(dst + C::KS_OFF + sa * kNB * 2, w.gks + sa * kNB * 2, (sb - sa) * kNB * 2, bar);
    bulk_g2s_w(dst + C::V_OFF + ra * C::VCODE, w.gv + ra * C::VCODE, (rb - ra) * C::VCODE, bar);
    bulk_g2s_w(dst + C::VS_OFF + sa * kNB * 2, w.gvs + sa * kNB * 2, (sb - sa) * kNB * 2, bar);
}

// Head-dim index of accumulator row rho (0..15) of PV m-tile mt = 2*block + h2.
template <int VT>
__device__ __forceinline__ int pv_dim(int mt, int rho)
{
    const int bb = mt >> 1, h2 = mt & 1, g = rho & 7, half = rho >> 3;
    if (VT == KVQ_V_Q4_0) return 32 * bb + 16 * h2 + 2 * g + half;
    return 32 * bb + 4 * g + 2 * h2 + half;
}

// PV A-fragment registers of one 32-block for the position pair (t, t+1):
// reg[h2][half] = fp16 pair (value at t, value at t+1) of the exact V code
// (q - 8 for q4_0, the int8 code for q8_0) of head dim pv_dim(2*bb + h2, g + 8*half).
// q4_0: w0 = [byte 2g of t, byte 2g+1 of t, byte 2g of t+1, byte 2g+1 of t+1]
// of the block (low nibbles = dims 2g, 2g+1, high = 2g+16, 2g+17).  q8_0:
// w0 = codes of dims 4g, 4g+1 and w1 of dims 4g+2, 4g+3, each as
// [t, t+1, t, t+1].
template <int VT>
__device__ __forceinline__ void v_pair_codes(uint32_t w0, uint32_t w1, uint32_t (&reg)[2][2])
{
    if (VT == KVQ_V_Q4_0) {
        const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));   // 1032
        const __half2 k16th = __half2half2(__ushort_as_half(0x2c00));   // 1/16
        const __half2 km72 = __half2half2(__ushort_as_half(0xd480));    // -72
        const uint32_t w23 = w0 >> 8;                                   // bytes 2g+1 at 0 and 2
        uint32_t x;
        x = (w0 & 0x000F000Fu) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&reg[0][0]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
        x = (w23 & 0x000F000Fu) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&reg[0][1]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
        x = (w0 & 0x00F000F0u) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&reg[1][0]) = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
        x = (w23 & 0x00F000F0u) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&reg[1][1]) = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
    } else {
        const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));   // 1152
        const uint32_t x0 = w0 ^ 0x80808080u, x1 = w1 ^ 0x80808080u;   // biased by 128
        uint32_t x;
        x = __byte_perm(x0, 0x64646464u, 0x4140);   // dim 4g
        *reinterpret_cast<__half2 *>(&reg[0][0]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x0, 0x64646464u, 0x4342);   // dim 4g+1
        *reinterpret_cast<__half2 *>(&reg[0][1]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x1, 0x64646464u, 0x4140);   // dim 4g+2
        *reinterpret_cast<__half2 *>(&reg[1][0]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x1, 0x64646464u, 0x4342);   // dim 4g+3
        *reinterpret_cast<__half2 *>(&reg[1][1]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
    }
}

__device__ __forceinline__ void unpack4h(uint2 raw, float (&x)[4])
{
    const float2 a = __half22float2(*reinterpret_cast<__half2 *>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<__half2 *>(&raw.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// Four signed int8 K codes -> two fp16 pairs holding 1152 + code (exact): the
// byte is biased by 128 (xor 0x80) and placed under the binary16 exponent of
// 1024 (0x64XX = 1024 + XX).
__device__ __forceinline__ void k_word_biased(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t x = w ^ 0x80808080u;
    lo = __byte_perm(x, 0x64646464u, 0x4140);
    hi = __byte_perm(x, 0x64646464u, 0x4342);
}

// Two signed int8 codes (bytes k0, k0+1 of w) -> exact fp16 pair.
__device__ __forceinline__ uint32_t q_pair(uint32_t w, int k0)
{
    const __half2 h = __halves2half2(__int2half_rn((int)(int8_t)(w >> (8 * k0))),
                                     __int2half_rn((int)(int8_t)(w >> (8 * k0 + 8))));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Kernel flavours (kModeDecode, kModeDump, kModeLoseStage of kvq_internal.cuh).
// In the lose-stage test flavour warp 0 of CTA 0 arms its second ring stage's
// barrier without issuing the stage's copies, so that this one wait (given a
// short limit) runs out and the give-up path runs: the warp skips that stage
// when it drains its copies, and waits with the normal limit for every copy
// it did issue, so no copy is in flight when the CTA exits.
constexpr int kLostStage = 1;                // issue index of the stage armed without copies
constexpr uint32_t kLostStageSpins = 1024;   // limit of the wait that runs out

template <int NT, int VT, int KT, int MODE, int W>
__global__ void __launch_bounds__(SplitCfg<NT, VT, KT, W>::THREADS, SplitCfg<NT, VT, KT, W>::MIN_CTAS)
    split_attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = SplitCfg<NT, VT, KT, W>;
    constexpr bool DUMP = MODE == kModeDump;
    constexpr bool LOSE = MODE == kModeLoseStage;
    static_assert(!(DUMP && KT == KVQ_K_F16), "the score dump exists for int8 K only");
    constexpr int kWarps = C::WARPS;
    constexpr int kThreads = C::THREADS;
    constexpr int S = C::STAGES;
    constexpr float kBias = 1152.0f;                 // K codes enter the MMA as 1152 + code
    // p = 2^(s - m) may reach 2^kSlack before m is raised; with the largest V
    // scale (65504 / 8) p * d then still fits fp16's range.
    constexpr float kSlack = 3.0f;
    extern __shared__ __align__(128) uint8_t smem[];

    // ---- the group, sequence, kv head and split of this CTA ----
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if ((int)blockIdx.x >= p.grp[k].cta0) gi = k;
    const GroupDesc &G = p.grp[gi];
    const int lb = (int)blockIdx.x - G.cta0;
    // row tile: rows [rt * 8NT, (rt + 1) * 8NT) of the kv head.  The 8-row
    // kernel is only chosen when every call of the launch has at most 8 rows
    // per kv head, so for it n_rt is 1 and row0 a constant 0.
    const int rt = (NT >= 2) ? lb % G.n_rt : 0, ls = (NT >= 2) ? lb / G.n_rt : lb;
    const int split = ls % G.n_split, h = (ls / G.n_split) % G.n_kv_heads, b = ls / G.n_split / G.n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int gb = p.grp_begin[G.head0 + h], gsz = p.grp_begin[G.head0 + h + 1] - gb;
    // This CTA's query rows: row0 + r (r < R) of the kv head's t_q x gsz rows,
    // row g being query token g / gsz of query head grp_q[gb + g % gsz].
    const int row0 = rt * 8 * NT;
    const int R = min(8 * NT, gsz * G.t_q - row0);
    if (R <= 0) return;   // a row tile past this kv head's rows (smaller group)
    const int seg0 = p.seq_seg0[G.seq0 + b], nseg = p.seq_nseg[G.seq0 + b];
    const int lcap = nseg ? min(G.max_len, p.seg[seg0 + nseg - 1].pos0 + p.seg[seg0 + nseg - 1].cap) : 0;
    // The split's positions as far as the segment table knows them: the
    // sequence length, read below, can only cut them shorter.  Copies of the
    // range go out before that read returns; positions at or past the length
    // are masked like any other invisible position.  Under the causal tail the
    // tile's last query token sees positions up to L - t_q + its index, and
    // L <= lcap bounds that from above.
    const int r0 = split * G.chunk;
    // (The clamp matters for long query chunks, which run on row tiles.)
    const int r1c = (NT >= 2) ? max(r0, min(min(lcap, r0 + G.chunk),
                                            G.causal ? lcap - G.t_q + (row0 + R - 1) / gsz + 1 : lcap))
                              : min(lcap, r0 + G.chunk);
    // The row tile holding the kv head's last query token sees every position
    // below L: it alone stores the appended tokens (fused append).
    const bool app_store = (NT >= 2) ? rt == (gsz * G.t_q - 1) / (8 * NT) : true;

    // Nothing above reads memory written by an earlier kernel.
    pdl_wait();
    pdl_trigger();
    const int len_b = G.seq_lens[b];

    // ---- the query rows' loads go out first: they are tiny, and issued after the
    // K/V prefetch below they would queue behind it ----
    constexpr int QPW = C::QROWS / kWarps;   // query rows per warp
    uint2 qraw[QPW];                          // all of this warp's row loads in flight at once
#pragma unroll
    for (int k = 0; k < QPW; ++k) {
        const int r = warp + kWarps * k;
        qraw[k] = make_uint2(0u, 0u);
        if (r < R && r0 < r1c) {
            const int i = (row0 + r) / gsz, hq = p.grp_q[gb + (row0 + r) % gsz];
            qraw[k] = *reinterpret_cast<const uint2 *>(G.q + (((size_t)b * G.t_q + i) * G.n_q_heads + hq) * kD + lane * 4);
        }
    }
    // ---- this warp's sub-range and its first copies (before the query prologue) ----
    const int span = (r1c - r0 + kWarps * kWTile - 1) / (kWarps * kWTile) * kWTile;
    const int w0 = min(r1c, r0 + warp * span), w1 = min(r1c, w0 + span);
    uint8_t *ring = smem + warp * C::RING;
    const uint32_t ring_s = smem_u32(ring);
    const uint32_t bar_s = smem_u32(smem + C::BAR_OFF) + warp * S * 8;
    int4 *tile_rec = reinterpret_cast<int4 *>(smem + C::TI_OFF) + warp * S;
    int *stage_n = reinterpret_cast<int *>(smem + C::NS_OFF) + warp * S;
    int *bad_flag = reinterpret_cast<int *>(smem + C::FLAG_OFF);
    if (tid == 0) *bad_flag = 0;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < S; ++st) mbar_init(bar_s + st * 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    Walk pw;
    walk_seek(p, seg0, nseg, h, w0, w1, 0, C::VCODE, pw, C::KCODE);
    int issued = 0;   // stages handed to the copy engine
    // Hand the next stage (up to TPS tiles of the current segment piece) to the
    // copy engine; the walk is advanced by every lane alike.
    // (test flavour) this warp arms one stage without its copies
    const bool loser = LOSE && blockIdx.x == 0 && warp == 0;
    auto issue = [&](int slot) {
        const int n = min(C::TPS, pw.Tend - pw.T);
        const int tb = pw.T * kWTile;
        if (lane == 0) {
            tile_rec[slot] = make_int4(tb, pw.la, pw.le, pw.pos0 + tb);
            stage_n[slot] = n | (pw.rows << 8);
        }
        // the whole warp from here (every condition is warp-uniform)
        if (loser && issued == kLostStage)
            mbar_arrive_expect_tx_w(bar_s + slot * 8, n * C::TILE);   // bytes that never come
        else if (pw.rows)   // rows layout: the piece's rows of these tiles only
            rows_issue<NT, VT, KT>(pw, max(pw.la, tb) - tb, min(pw.le, tb + n * kWTile) - tb,
                                   ring_s + slot * C::STAGE, bar_s + slot * 8);
        else
            tile_issue<NT, VT, KT>(pw, n, ring_s + slot * C::STAGE, bar_s + slot * 8);
        pw.T += n;
        pw.gk += n * C::TILE_K;
        pw.gks += n * C::TILE_S;
        pw.gv += n * C::TILE_V;
        pw.gvs += n * C::TILE_S;
        if (pw.T >= pw.Tend) walk_seek(p, seg0, nseg, h, w0, w1, pw.k + 1, C::VCODE, pw, C::KCODE);
        ++issued;
    };
#pragma unroll
    for (int st = 0; st < S - 1; ++st)
        if (pw.k < nseg) issue(st);

    const int L = max(0, min(len_b, lcap));
    const int r1 = min(min(L, r0 + G.chunk), r1c);
    if (r0 >= r1) {                                  // no position in this split
        for (int j = 0; j < issued; ++j) mbar_wait(bar_s + (j % S) * 8, (j / S) & 1);
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

    // ---- tokens this call appends that fall in this split (fused append):
    // quantized by the append rules, stored to the open segment for later calls
    // and kept in shared memory to patch into this call's staged tiles ----
    int na0 = 0, nn = 0;   // absolute positions [na0, na0 + nn)
    uint32_t *newrow = reinterpret_cast<uint32_t *>(smem + C::NEW_OFF);
    if (G.k_new != nullptr) {
        const int ap = p.app_pos[G.seq0 + b];
        const int lo = max(ap, r0), hi = min(ap + G.t_q, r0 + G.chunk);
        if (lo < hi) {
            na0 = lo;
            nn = hi - lo;
        }
        const SegDesc &sl = p.seg[seg0 + nseg - 1];   // the open segment
        for (int i = warp; i < nn; i += kWarps) {
            const size_t src = (((size_t)b * G.t_q + (na0 + i - ap)) * G.n_kv_heads + h) * kD;
            const TokenRow t = quant_token<VT>(G.k_new + src, G.v_new + src, lane);
            const int local = na0 + i - sl.pos0, u = local % kWTile;
            const size_t tile = (size_t)h * sl.cap + local - u;
            if (app_store && sl.layout == KVQ_LAYOUT_ROWS)
                store_token_rows<VT>(t, lane, const_cast<uint8_t *>(sl.kq) + (tile + u) * kD,
                                     const_cast<uint16_t *>(sl.ks) + (tile + u) * kNB,
                                     const_cast<uint8_t *>(sl.vq) + (tile + u) * C::VCODE,
                                     const_cast<uint16_t *>(sl.vs) + (tile + u) * kNB);
            else if (app_store)
                store_token<VT>(t, u, lane, const_cast<uint8_t *>(sl.kq) + tile * kD,
                                const_cast<uint16_t *>(sl.ks) + (tile + u) * kNB,
                                const_cast<uint8_t *>(sl.vq) + tile * C::VCODE,
                                const_cast<uint16_t *>(sl.vs) + (tile + u) * kNB);
            newrow[(i * 32 + lane) * 3 + 0] = t.kw;
            newrow[(i * 32 + lane) * 3 + 1] = t.vw;
            newrow[(i * 32 + lane) * 3 + 2] = (uint32_t)t.ks | ((uint32_t)t.vs << 16);
        }
    }

    uint4 *qf = reinterpret_cast<uint4 *>(smem + C::QF_OFF) + lane;   // chunk k at qf[32 * k]
    if constexpr (KT == KVQ_K_F16) {
        // ---- F16 K: the query rows stay fp16 (not quantized).  k16 step ks of
        // 8-row tile nt takes B registers (dims 16ks + 2c, +1 | 16ks + 2c + 8, +9)
        // of row 8nt + g: words 8ks + c and 8ks + c + 4 of the row; chunk
        // nt * 4 + ks/2 holds steps 2kp, 2kp + 1 ----
        uint32_t *qh = reinterpret_cast<uint32_t *>(smem + C::Q_OFF);   // [QROWS][64 words]
#pragma unroll
        for (int k = 0; k < QPW; ++k) {
            const int r = warp + kWarps * k;
            qh[r * (kD / 2) + 2 * lane] = qraw[k].x;
            qh[r * (kD / 2) + 2 * lane + 1] = qraw[k].y;
        }
        __syncthreads();
        for (int k = warp; k < NT * 4; k += kWarps) {
            const int nt = k / 4, kp = k % 4;
            const uint32_t *w = qh + (8 * nt + g) * (kD / 2) + 16 * kp + c;
            qf[32 * k] = make_uint4(w[0], w[4], w[8], w[12]);
        }
    } else {
        // ---- quantize the query rows of this kv head (int8 rule, fp16 scale) ----
        uint32_t *qw = reinterpret_cast<uint32_t *>(smem + C::Q_OFF);
        float *qs = reinterpret_cast<float *>(smem + C::QS_OFF);
        int *qsum = reinterpret_cast<int *>(smem + C::QSUM_OFF);
    #pragma unroll
        for (int k = 0; k < QPW; ++k) {
            const int r = warp + kWarps * k;
            uint32_t word = 0;
            float s = 0.f;
            int sum = 0;
            if (r < R) {
                const int i = (row0 + r) / gsz, hq = p.grp_q[gb + (row0 + r) % gsz];
                const size_t qrow = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
                float x[4];
                unpack4h(qraw[k], x);
                float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
                const __half sh = __float2half_rn(__fdiv_rn(a, 127.f));
                s = __half2float(sh);
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int code = quant_i8(x[k], s);
                    word |= (uint32_t)(code & 0xff) << (8 * k);
                    sum += code;
                }
                if (DUMP && split == 0) {
                    reinterpret_cast<uint32_t *>(G.dbg_qc)[qrow * (kD / 4) + lane] = word;
                    if ((lane & 7) == 0) G.dbg_qs[qrow * kNB + (lane >> 3)] = __half_as_ushort(sh);
                }
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            qw[r * (kD / 4) + lane] = word;
            if ((lane & 7) == 0) {
                qs[r * kNB + (lane >> 3)] = s * G.qk_scale_log2;
                qsum[r * kNB + (lane >> 3)] = sum;
            }
        }
        __syncthreads();   // query codes visible

        // Query B fragments (fp16, exact codes).  Within block bb, k16 step ks, this
        // lane's k slots (2c, 2c+1 | 2c+8, 2c+9) carry head dims
        // 32bb + 8c + 4ks + (0, 1 | 2, 3): the bytes of word 8bb + 2c + ks, the same
        // word the lane reads from K, so q.k is unchanged.  The warps write them, with
        // the accumulator seeds (-1152 * sum of the row's codes in the block) of
        // rows 2c, 2c+1 and those rows' scales, to the per-lane table that every
        // stage reads back (row scales as (row 2c, row 2c+1) pairs per block).
        // (nt, block) entries are spread over the warps: entry k goes to warp k % WARPS.
        for (int k = warp; k < NT * kNB + NT * 2; k += kWarps) {
            if (k < NT * kNB) {
                const int nt = k / kNB, bb = k % kNB;
                const uint32_t w0 = qw[(8 * nt + g) * (kD / 4) + 8 * bb + 2 * c];
                const uint32_t w1 = qw[(8 * nt + g) * (kD / 4) + 8 * bb + 2 * c + 1];
                qf[32 * (nt * kNB + bb)] = make_uint4(q_pair(w0, 0), q_pair(w0, 2), q_pair(w1, 0), q_pair(w1, 2));
                const float s0 = -kBias * (float)qsum[(8 * nt + 2 * c) * kNB + bb];
                const float s1 = -kBias * (float)qsum[(8 * nt + 2 * c + 1) * kNB + bb];
                qf[32 * (C::QB_CHUNKS + nt * kNB + bb)] =
                    make_uint4(__float_as_uint(s0), __float_as_uint(s1), __float_as_uint(s0), __float_as_uint(s1));
            } else {
                // (row 2c, row 2c+1) scale pairs of blocks 2hb, 2hb+1
                const int nt = (k - NT * kNB) / 2, hb = (k - NT * kNB) % 2;
                const int r0 = 8 * nt + 2 * c;
                qf[32 * (C::QB_CHUNKS + C::SEED_CHUNKS + nt * 2 + hb)] =
                    make_uint4(__float_as_uint(qs[r0 * kNB + 2 * hb]), __float_as_uint(qs[(r0 + 1) * kNB + 2 * hb]),
                               __float_as_uint(qs[r0 * kNB + 2 * hb + 1]), __float_as_uint(qs[(r0 + 1) * kNB + 2 * hb + 1]));
            }
        }
    }
    __syncthreads();   // query table visible
    // This lane's rows are 8nt + 2c + e (e = 0, 1): the columns of its QK
    // accumulators and of its P.V accumulators alike.
    float m[NT][2], l[NT][2];
    int lim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int row = 8 * nt + 2 * c + e;
            lim[nt][e] = (row < R) ? (G.causal ? L - G.t_q + (row0 + row) / gsz : L - 1) : -1;
            m[nt][e] = -INFINITY;
            l[nt][e] = 0.f;
        }
    float2 mu[NT];   // exponent offsets: m, or 0 while m is -inf
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mu[nt] = make_float2(0.f, 0.f);
    const int lim_min = G.causal ? L - G.t_q + row0 / gsz : L - 1;   // smallest limit over live rows
    float acc[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[mt][nt][k] = 0.f;

    bool bad = false;   // a stage never arrived (the warp then stops and drains)
    int slot = 0, phase = 0, prev = S - 1, done = 0;   // done % S, (done / S) & 1, (done + S - 1) % S
    while (done < issued) {
        const bool landed = (loser && done == kLostStage) ? mbar_wait(bar_s + slot * 8, phase, kLostStageSpins)
                                                          : mbar_wait(bar_s + slot * 8, phase);
        if (!__all_sync(0xffffffffu, landed)) {
            bad = true;
            break;
        }
        __syncwarp();   // every lane is done with the previous stage, whose slot is refilled next
        if (pw.k < nseg) {
            // every lane (the elected issuing lane among them): the lanes'
            // generic reads of the slot before the copy engine's writes
            fence_proxy_async_smem();
            issue(prev);
        }
        const int ns = stage_n[slot] & 0xff;
        const uint8_t *stg = ring + slot * C::STAGE;
        const int4 rec0 = tile_rec[slot];
        if (KT == KVQ_K_I8 && (stage_n[slot] >> 8)) {   // rows layout: permute the staged tiles into the tile order
            for (int t = 0; t < ns; ++t) {
                rows_to_tile_k(const_cast<uint8_t *>(stg) + C::K_OFF + t * C::TILE_K, lane);
                rows_to_tile_v<VT>(const_cast<uint8_t *>(stg) + C::V_OFF + t * C::TILE_V, lane);
            }
        }
        prev = slot;
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        ++done;
#pragma unroll 1
        for (int t = 0; t < ns; ++t) {
        const uint8_t *stK = stg + C::K_OFF + t * C::TILE_K, *stKS = stg + C::KS_OFF + t * C::TILE_S;
        const uint8_t *stV = stg + C::V_OFF + t * C::TILE_V, *stVS = stg + C::VS_OFF + t * C::TILE_S;
        const int tb = rec0.x + t * kWTile, la = rec0.y, le = rec0.z, pos_base = rec0.w + t * kWTile;
        // every position of the tile valid and visible to every live row?
        const bool full = tb >= la && tb + kWTile <= le && pos_base + kWTile - 1 <= lim_min;
        if (nn > 0 && pos_base < na0 + nn && pos_base + kWTile > na0) {
            // this call's appended tokens: the staged copy may predate their
            // store, so write their rows into the stage
            for (int a = max(na0, pos_base); a < min(na0 + nn, pos_base + kWTile); ++a) {
                const int i = a - na0;
                TokenRow t;
                t.kw = newrow[(i * 32 + lane) * 3 + 0];
                t.vw = newrow[(i * 32 + lane) * 3 + 1];
                const uint32_t sv = newrow[(i * 32 + lane) * 3 + 2];
                t.ks = (uint16_t)(sv & 0xffffu);
                t.vs = (uint16_t)(sv >> 16);
                const int u = a - pos_base;
                store_token<VT>(t, u, lane, const_cast<uint8_t *>(stK), reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(stKS)) + u * kNB,
                                const_cast<uint8_t *>(stV), reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(stVS)) + u * kNB);
            }
            __syncwarp();
        }

        auto chunk = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            float2 s[NT][2];   // [nt][position g / g + 8] = (row 2c, row 2c + 1)
            if constexpr (KT == KVQ_K_F16) {
                // ---- S^T = K Q^T over the fp16 values: A = the K tile's 16
                // positions (one 16-byte fragment load per k16 step), B = 8
                // query rows, fp32 accumulation ----
                float sc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) sc[nt][k] = 0.f;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint4 a4 = *reinterpret_cast<const uint4 *>(stK + ks * 512 + lane * 16);
                    const uint32_t av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint4 qb = qf[32 * (nt * 4 + ks / 2)];
                        mma_f16_16816(sc[nt], av, (ks & 1) ? qb.z : qb.x, (ks & 1) ? qb.w : qb.y);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        float2 a = mul2(make_float2(sc[nt][2 * pp], sc[nt][2 * pp + 1]),
                                        make_float2(G.qk_scale_log2, G.qk_scale_log2));
                        if (!FULL) {
                            const int tok = tb + 8 * pp + g, pos = pos_base + 8 * pp + g;
                            const bool okp = tok >= la && tok < le;
                            a.x = (okp && pos <= lim[nt][0]) ? a.x : -INFINITY;
                            a.y = (okp && pos <= lim[nt][1]) ? a.y : -INFINITY;
                        }
                        s[nt][pp] = a;
                    }
            } else {
                // ---- S^T = K Q^T per 32-block (exact integers in fp32): A = the K
                // codes of the stage's 16 positions (rows g and g + 8 of the MMA),
                // B = 8 query rows ----
                uint4 kk[2][2];   // [position g / g + 8][blocks 0-1 / 2-3]
    #pragma unroll
                for (int pp = 0; pp < 2; ++pp)
    #pragma unroll
                    for (int hb = 0; hb < 2; ++hb)
                        kk[pp][hb] = *reinterpret_cast<const uint4 *>(stK + (2 * pp + hb) * 512 + lane * 16);
                float sc[NT][kNB][4];   // (pos g, row 2c), (pos g, row 2c+1), (pos g+8, row 2c), (pos g+8, row 2c+1)
    #pragma unroll
                for (int bb = 0; bb < kNB; ++bb) {
                    const uint4 &u0 = kk[0][bb >> 1], &u1 = kk[1][bb >> 1];
                    uint32_t a0[4], a1[4];   // k16 steps 0 and 1 of the block
                    k_word_biased((bb & 1) ? u0.z : u0.x, a0[0], a0[2]);
                    k_word_biased((bb & 1) ? u1.z : u1.x, a0[1], a0[3]);
                    k_word_biased((bb & 1) ? u0.w : u0.y, a1[0], a1[2]);
                    k_word_biased((bb & 1) ? u1.w : u1.y, a1[1], a1[3]);
    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint4 qb = qf[32 * (nt * kNB + bb)];
                        const uint4 sd = qf[32 * (C::QB_CHUNKS + nt * kNB + bb)];
                        mma_f16_16816_c4(sc[nt][bb], a0, qb.x, qb.y, sd);
                        mma_f16_16816(sc[nt][bb], a1, qb.z, qb.w);
                    }
                }
                // K scales of this lane's positions g and g + 8
                float sk[2][kNB];
                unpack4h(*reinterpret_cast<const uint2 *>(stKS + g * kNB * 2), sk[0]);
                unpack4h(*reinterpret_cast<const uint2 *>(stKS + (g + 8) * kNB * 2), sk[1]);
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float2 sq[kNB];   // (row 2c, row 2c + 1) scales of each block
    #pragma unroll
                    for (int hb = 0; hb < 2; ++hb) {
                        const uint4 q4 = qf[32 * (C::QB_CHUNKS + C::SEED_CHUNKS + nt * 2 + hb)];
                        sq[2 * hb] = make_float2(__uint_as_float(q4.x), __uint_as_float(q4.y));
                        sq[2 * hb + 1] = make_float2(__uint_as_float(q4.z), __uint_as_float(q4.w));
                    }
    #pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        float2 a = make_float2(0.f, 0.f);
    #pragma unroll
                        for (int bb = 0; bb < kNB; ++bb) {
                            const float2 i2 = make_float2(sc[nt][bb][2 * pp], sc[nt][bb][2 * pp + 1]);
                            a = fma2(mul2(i2, sq[bb]), make_float2(sk[pp][bb], sk[pp][bb]), a);
                        }
                        if (!FULL) {
                            const int tok = tb + 8 * pp + g, pos = pos_base + 8 * pp + g;
                            const bool okp = tok >= la && tok < le;
                            a.x = (okp && pos <= lim[nt][0]) ? a.x : -INFINITY;
                            a.y = (okp && pos <= lim[nt][1]) ? a.y : -INFINITY;
                        }
                        s[nt][pp] = a;
                    }
                }
                if constexpr (DUMP) {
    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
    #pragma unroll
                        for (int pp = 0; pp < 2; ++pp)
    #pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int row = 8 * nt + 2 * c + e, tok = tb + 8 * pp + g, pos = pos_base + 8 * pp + g;
                                if (row < R && tok >= la && tok < le && pos < L) {
                                    const int i = (row0 + row) / gsz, hq = p.grp_q[gb + (row0 + row) % gsz];
                                    const size_t o = ((((size_t)b * G.t_q + i) * G.n_q_heads + hq) * G.max_len + pos) * kNB;
                                    int4 v;
                                    v.x = (int)sc[nt][0][2 * pp + e]; v.y = (int)sc[nt][1][2 * pp + e];
                                    v.z = (int)sc[nt][2][2 * pp + e]; v.w = (int)sc[nt][3][2 * pp + e];
                                    *reinterpret_cast<int4 *>(G.dbg_scores + o) = v;
                                }
                            }
                    return;
                }
            }

            // ---- online softmax (base 2) with a lazily raised reference max: a
            // row's 16 scores sit in the 8 lanes of one c, and the exact max over
            // them (three shuffles) is only taken when some score exceeds the
            // row's reference by more than kSlack, so p stays <= 2^kSlack ----
            bool need = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                need |= fmaxf(s[nt][0].x, s[nt][1].x) > m[nt][0] + kSlack;
                need |= fmaxf(s[nt][0].y, s[nt][1].y) > m[nt][1] + kSlack;
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float al[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float mx = e ? fmaxf(s[nt][0].y, s[nt][1].y) : fmaxf(s[nt][0].x, s[nt][1].x);
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float mnew = fmaxf(m[nt][e], mx);
                        al[e] = (mnew == -INFINITY) ? 1.f : fast_exp2(m[nt][e] - mnew);
                        l[nt][e] *= al[e];
                        m[nt][e] = mnew;
                    }
                    mu[nt] = make_float2(m[nt][0] == -INFINITY ? 0.f : m[nt][0], m[nt][1] == -INFINITY ? 0.f : m[nt][1]);
                    const float2 a2 = make_float2(al[0], al[1]);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const float2 lo = mul2(make_float2(acc[mt][nt][0], acc[mt][nt][1]), a2);
                        const float2 hi = mul2(make_float2(acc[mt][nt][2], acc[mt][nt][3]), a2);
                        acc[mt][nt][0] = lo.x; acc[mt][nt][1] = lo.y;
                        acc[mt][nt][2] = hi.x; acc[mt][nt][3] = hi.y;
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const float2 t = sub2(s[nt][pp], mu[nt]);
                    s[nt][pp] = make_float2(fast_exp2(t.x), fast_exp2(t.y));
                    lsum = add2(lsum, s[nt][pp]);
                }
                l[nt][0] += lsum.x;
                l[nt][1] += lsum.y;
            }

            // ---- O += P . V  (per 32-block: A = V codes, B = p*d as fp16 hi + lo,
            // formed at (position, row) and transposed to (row, position) with
            // movmatrix) ----
            float dv[2][kNB];   // V scales of positions g, g + 8 (0 where invisible)
            unpack4h(*reinterpret_cast<const uint2 *>(stVS + g * kNB * 2), dv[0]);
            unpack4h(*reinterpret_cast<const uint2 *>(stVS + (g + 8) * kNB * 2), dv[1]);
            if (!FULL) {
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const int tok = tb + 8 * pp + g;
                    const bool ok = tok >= la && tok < le && pos_base + 8 * pp + g < L;
#pragma unroll
                    for (int bb = 0; bb < kNB; ++bb) dv[pp][bb] = ok ? dv[pp][bb] : 0.f;
                }
            }
            // V code words of positions (8sub + 2c, +1): q4_0 one load per sub
            // (word bb = block bb), q8_0 two (load 2sub + hb: blocks 2hb, 2hb + 1)
            constexpr int NVL = (VT == KVQ_V_Q4_0) ? 1 : 2;
            uint4 vv[2][NVL];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub)
#pragma unroll
                for (int hb = 0; hb < NVL; ++hb)
                    vv[sub][hb] = *reinterpret_cast<const uint4 *>(stV + (NVL * sub + hb) * 512 + lane * 16);
#pragma unroll
            for (int bb = 0; bb < kNB; ++bb) {
                uint32_t a[2][4];   // [h2] A fragment of m-tile 2bb + h2
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    uint32_t r[2][2];
                    if (VT == KVQ_V_Q4_0) {
                        const uint4 &v = vv[sub][0];
                        v_pair_codes<VT>(bb == 0 ? v.x : bb == 1 ? v.y : bb == 2 ? v.z : v.w, 0u, r);
                    } else {
                        const uint4 &v = vv[sub][NVL - 1 == 0 ? 0 : (bb >> 1)];
                        v_pair_codes<VT>((bb & 1) ? v.z : v.x, (bb & 1) ? v.w : v.y, r);
                    }
                    a[0][2 * sub] = r[0][0];
                    a[0][2 * sub + 1] = r[0][1];
                    a[1][2 * sub] = r[1][0];
                    a[1][2 * sub + 1] = r[1][1];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t bh[2], bl[2];   // [positions 0-7 / 8-15]
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        // x = p*d split as hi = fp16(x) (rounded) + lo = fp16(x - hi), with
                        // x - hi exact in fp32: about 22 bits of x survive
                        const float2 x = mul2(s[nt][pp], make_float2(dv[pp][bb], dv[pp][bb]));
                        const uint32_t hp = pack_half2(x.x, x.y);
                        const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hp));
                        const float2 lo = sub2(x, h);
                        bh[pp] = movmatrix_t(hp);
                        bl[pp] = movmatrix_t(pack_half2(lo.x, lo.y));
                    }
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        mma_f16_16816(acc[2 * bb + h2][nt], a[h2], bh[0], bh[1]);
                        mma_f16_16816(acc[2 * bb + h2][nt], a[h2], bl[0], bl[1]);
                    }
                }
            }
        };
        if (full)
            chunk(std::integral_constant<bool, true>());
        else
            chunk(std::integral_constant<bool, false>());
        }
    }

    if (bad) {
        // a wait gave up: wait (bounded) for this warp's copies still in flight,
        // then poison the CTA's results
        for (int j = done; j < issued; ++j)
            if (!(loser && j == kLostStage)) mbar_wait(bar_s + (j % S) * 8, (j / S) & 1);
        if (lane == 0) {
            atomicOr(bad_flag, 1);
            atomicAdd(p.timeouts, 1u);
        }
    }
    if constexpr (!DUMP) {
        // ---- merge the warps' (m, l, acc) in a fixed order and write ----
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 4);
                l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 8);
                l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], 16);
            }
        __syncthreads();   // every warp is done with the stage rings
        constexpr int RW = 8 * NT;                          // rows per warp state
        float *sm_m = reinterpret_cast<float *>(smem + C::ML_OFF);   // [warp][RW]
        float *sm_l = sm_m + kWarps * RW;
        float *sm_M = sm_l + kWarps * RW, *sm_inv = sm_M + RW, *sm_lse = sm_inv + RW;   // [RW]
        float *sm_o = reinterpret_cast<float *>(smem);      // slices [warp][RW][OROW]
        if (g == 0)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sm_m[warp * RW + 8 * nt + 2 * c + e] = m[nt][e];
                    sm_l[warp * RW + 8 * nt + 2 * c + e] = l[nt][e];
                }
        __syncthreads();
        if (tid < R) {   // row totals: M = max_w m_w, L = sum_w l_w 2^(m_w - M)
            float M = -INFINITY;
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * RW + tid]);
            float Lsum = 0.f;
            for (int w = 0; w < kWarps; ++w) {
                const float mw = sm_m[w * RW + tid];
                if (mw != -INFINITY) Lsum += sm_l[w * RW + tid] * fast_exp2(mw - M);
            }
            float inv, lg;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(Lsum));
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(Lsum));
            const bool any = Lsum > 0.f;
            sm_M[tid] = M;
            sm_inv[tid] = any ? inv : 0.f;
            sm_lse[tid] = any ? (M + lg) * 0.69314718055994531f : -INFINITY;
        }
        __syncthreads();
        // Each (row, dim) belongs to one lane per warp; a warp's accumulator is
        // scaled by 2^(m_warp - M) / L.  Head dims pv_dim(mt, g) and
        // pv_dim(mt, g + 8) are adjacent, so a lane stores them as one pair.
        constexpr bool kSlices = C::SLICES;
        auto put = [&](float *dst, bool add) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = 8 * nt + 2 * c + e;
                    if (row >= R) continue;
                    const float mw = m[nt][e];
                    const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - sm_M[row]) * sm_inv[row];
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        float2 *o = reinterpret_cast<float2 *>(&dst[row * C::OROW + pv_dim<VT>(mt, g)]);
                        float2 v = make_float2(acc[mt][nt][e] * f, acc[mt][nt][2 + e] * f);
                        if (add) {
                            const float2 q = *o;
                            v.x += q.x;
                            v.y += q.y;
                        }
                        *o = v;
                    }
                }
        };
        if (kSlices) {
            put(sm_o + warp * RW * C::OROW, false);
            __syncthreads();
        } else {
            // warp 0 stores, the others add in turn
            for (int w = 0; w < kWarps; ++w) {
                if (warp == w) put(sm_o, w > 0);
                __syncthreads();
            }
        }
        const bool poisoned = *bad_flag != 0;   // set before the merge's first barrier
        for (int i4 = tid; i4 < R * (kD / 4); i4 += kThreads) {
            const int row = i4 / (kD / 4), d = (i4 % (kD / 4)) * 4;
            float4 t = *reinterpret_cast<const float4 *>(&sm_o[row * C::OROW + d]);
            if (kSlices) {
#pragma unroll
                for (int w = 1; w < kWarps; ++w) {
                    const float4 q = *reinterpret_cast<const float4 *>(&sm_o[(w * RW + row) * C::OROW + d]);
                    t.x += q.x; t.y += q.y; t.z += q.z; t.w += q.w;
                }
            }
            float ls = sm_lse[row];
            if (poisoned) t.x = t.y = t.z = t.w = ls = __int_as_float(0x7fc00000);   // NaN: the CTA lost a stage
            const int i = (row0 + row) / gsz, hq = p.grp_q[gb + (row0 + row) % gsz];
            const size_t orow = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
            if (G.n_split == 1) {
                *reinterpret_cast<float4 *>(G.out + orow * kD + d) = t;
                if (d == 0) G.lse[orow] = ls;
            } else {
                *reinterpret_cast<float4 *>(G.ws_o + (orow * G.n_split + split) * kD + d) = t;
                if (d == 0) G.ws_lse[orow * G.n_split + split] = ls;
            }
        }
    }
}

template <int NT, int VT, int KT, int W>
cudaError_t launch_split_t(const AttnParams &p, int n_ctas, int mode, cudaStream_t s, bool pdl)
{
    using C = SplitCfg<NT, VT, KT, W>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if constexpr (KT == KVQ_K_I8 && W == split_warps(NT)) {
        if (mode == kModeDump) return cudaLaunchKernelEx(&cfg, split_attn_kernel<NT, VT, KT, kModeDump, W>, p);
    }
    if constexpr (KT == KVQ_K_I8 && VT == KVQ_V_Q4_0 && NT == 1 && W == split_warps(1)) {
        if (mode == kModeLoseStage)
            return cudaLaunchKernelEx(&cfg, split_attn_kernel<NT, VT, KT, kModeLoseStage, W>, p);
    }
    if (mode != kModeDecode) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, split_attn_kernel<NT, VT, KT, kModeDecode, W>, p);
}

template <int NT, int VT, int KT, int W>
cudaError_t prepare_split_t(int mode, int *ctas_per_sm)
{
    using C = SplitCfg<NT, VT, KT, W>;
    const void *fn = nullptr;
    if (mode == kModeDecode) fn = (const void *)split_attn_kernel<NT, VT, KT, kModeDecode, W>;
    if constexpr (KT == KVQ_K_I8 && W == split_warps(NT)) {
        if (mode == kModeDump) fn = (const void *)split_attn_kernel<NT, VT, KT, kModeDump, W>;
    }
    if constexpr (KT == KVQ_K_I8 && VT == KVQ_V_Q4_0 && NT == 1 && W == split_warps(1)) {
        if (mode == kModeLoseStage) fn = (const void *)split_attn_kernel<NT, VT, KT, kModeLoseStage, W>;
    }
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (ctas_per_sm) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, C::THREADS, C::SMEM);
    return cudaSuccess;
}

template <int VT, int KT>
cudaError_t launch_split_nt(const AttnParams &p, int nt, int warps, int n_ctas, int mode, cudaStream_t s, bool pdl)
{
    if (nt == 1 && warps == kWarpsHalf) return launch_split_t<1, VT, KT, kWarpsHalf>(p, n_ctas, mode, s, pdl);
    if (warps != split_warps(nt)) return cudaErrorInvalidValue;
    switch (nt) {
    case 1: return launch_split_t<1, VT, KT, split_warps(1)>(p, n_ctas, mode, s, pdl);
    case 2: return launch_split_t<2, VT, KT, split_warps(2)>(p, n_ctas, mode, s, pdl);
    case 4: return launch_split_t<4, VT, KT, split_warps(4)>(p, n_ctas, mode, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <int VT, int KT>
cudaError_t prepare_split_nt(int nt, int warps, int mode, int *ctas)
{
    if (nt == 1 && warps == kWarpsHalf) return prepare_split_t<1, VT, KT, kWarpsHalf>(mode, ctas);
    if (warps != split_warps(nt)) return cudaErrorInvalidValue;
    switch (nt) {
    case 1: return prepare_split_t<1, VT, KT, split_warps(1)>(mode, ctas);
    case 2: return prepare_split_t<2, VT, KT, split_warps(2)>(mode, ctas);
    case 4: return prepare_split_t<4, VT, KT, split_warps(4)>(mode, ctas);
    default: return cudaErrorInvalidValue;
    }
}

#define KVQ_DEFINE_SPLIT_ENTRY(SUFFIX, VT)                                                              \
    cudaError_t launch_split_##SUFFIX(const AttnParams &p, int nt, int warps, int k_type, int n_ctas,    \
                                      int mode, cudaStream_t s, bool pdl)                               \
    {                                                                                                   \
        return (k_type == KVQ_K_F16) ? launch_split_nt<VT, KVQ_K_F16>(p, nt, warps, n_ctas, mode, s, pdl) \
                                     : launch_split_nt<VT, KVQ_K_I8>(p, nt, warps, n_ctas, mode, s, pdl); \
    }                                                                                                   \
    cudaError_t prepare_split_##SUFFIX(int nt, int warps, int k_type, int mode, int *ctas)              \
    {                                                                                                   \
        return (k_type == KVQ_K_F16) ? prepare_split_nt<VT, KVQ_K_F16>(nt, warps, mode, ctas)           \
                                     : prepare_split_nt<VT, KVQ_K_I8>(nt, warps, mode, ctas);           \
    }

}  // namespace kvq
