// kvq_verify.cuh -- attention over the quantized cache for calls with 9 to 32
// query rows per kv head (multi-token verify: t_q query tokens x the query
// heads of a kv head) on the sm_103a tensor cores, with the cache positions on
// the MMA's M dimension and the query rows on N.
//
// One CTA = (split s, kv head h, sequence b) of a work group, indexed like the
// split kernel's CTAs (one row tile): it attends the kv head's R <= 32 query
// rows over the positions [s*chunk, (s+1)*chunk) of sequence b, 128 positions
// (one KV tile) at a time, and writes the final output (one split) or a
// partial (normalised o, lse) for the combine kernel.
//
// The arithmetic is the split kernel's (per-32 int8 K and Q with fp16 scales,
// exact integer block dot, q4_0 / q8_0 V), laid out transposed:
//   * S_b^T = K_b Q_b^T per 32-block b: A = the tile's K codes as exact fp16
//     integers (128 positions x 32 dims, K-major), B = the query codes (32 rows,
//     K-major), two K = 16 steps into one TMEM accumulator per block (lane =
//     position, column = row); every partial sum is an integer below 2^24.
//     score = sum_b S_b * (sq_b * sm_scale * log2 e) * sk_b.
//   * online softmax in base 2: one thread per (position, 16 rows); the rows'
//     reference maxima are shared by the four warps that hold a row half and
//     raised only when a score passes them by more than 3 (p <= 8); a raise
//     takes the exact tile maximum of each row (a butterfly over the warp and
//     an exchange between the four warps) and rescales O.
//   * O^T += V^T P^T: A = the tile's V as v / 2 = code * (d / 2) split into
//     fp16 hi and lo (dims x positions, K-major), B = p split into fp16 hi and
//     lo (rows x positions, stored MN-major: each position's 8 rows side by
//     side), three MMAs per 16 positions (hi.hi, hi.lo, lo.hi), ~22 bits of
//     every product; O^T in TMEM (lane = head dim, column = row).
//
// Warp roles (512 threads):
//   warps 0-7   softmax: warp w holds TMEM lane quarter w % 4 (positions
//               32(w%4).. of a tile, head dims 32(w%4).. of O^T) and rows
//               16(w/4)..16(w/4)+15; the final O^T read-out.  Lane 0 of warp
//               0 also issues the P.V MMAs of each tile once every softmax
//               warp has written its P, and walks the segments and issues the
//               bulk copies of the tiles RS ahead;
//   warps 8-11  K converters: K codes and K scales of a tile to the K operand;
//               lane 0 of warp 8 issues the tile's QK MMAs;
//   warps 12-15 V converters: V codes of a tile, half by half (64 positions),
//               to the V hi / lo operands.
// Every wait is bounded: a wait that gives up marks the CTA, the roles leave
// their loops, in-flight copies and MMAs are waited for (bounded), TMEM is
// released and the CTA's rows are written as NaN.
#pragma once

#include "kvq_prefill.cuh"

namespace kvq {

constexpr int kVM = kVerifyPositions;    // positions per KV tile (MMA M of QK^T, K extent of P.V): 128
constexpr int kVN = kVerifyRows;         // query rows per CTA (MMA N): 32
constexpr int kVSub = kVM / kWTile;      // cache tiles per KV tile (8)
constexpr int kVHalf = kVM / 2;          // positions per V operand half (64)
constexpr int kVSoftWarps = 8;           // warp 0's lane 0 also issues the P.V MMAs and the bulk copies
constexpr int kVKWarp0 = 8;              // four K converter warps; lane 0 of the first issues the QK MMAs
constexpr int kVKWarps = 4;
constexpr int kVVWarp0 = 12;             // four V converter warps
constexpr int kVWarps = 16;
constexpr int kVThreads = kVWarps * 32;
static_assert(kVN == 32, "the softmax warps hold two halves of 16 rows");

template <int VT>
struct VerifyCfg {
    static constexpr int VCODE = (VT == KVQ_V_Q4_0) ? kD / 2 : kD;
    static constexpr int TILE_K = kWTile * kD, TILE_S = kWTile * kNB * 2, TILE_V = kWTile * VCODE;
    static constexpr int RS = (VT == KVQ_V_Q4_0) ? 3 : 2;           // raw stages
    static constexpr int R_K = 0, R_KS = R_K + kVSub * TILE_K, R_V = R_KS + kVSub * TILE_S;
    static constexpr int R_VS = R_V + kVSub * TILE_V, RAW = R_VS + kVSub * TILE_S;
    static constexpr int TILE = TILE_K + TILE_S + TILE_V + TILE_S;
    // K operand [128 positions][128 dims], K-major: 8-position row groups of 16
    // core matrices K_LBO apart (160: the converters' stores are conflict free)
    static constexpr int K_LBO = 160, K_SBO = 16 * K_LBO, KBUF = (kVM / 8) * K_SBO;
    // V operand half [128 dims][64 positions], K-major, 8-dim row groups padded
    static constexpr int V_SBO = (kVHalf / 8) * 128 + 16, VBUF = (kD / 8) * V_SBO;
    // Q operand [32 rows][128 dims], K-major
    static constexpr int Q_SBO = 16 * 128, QBUF = (kVN / 8) * Q_SBO;
    // P operand [128 positions][32 rows], MN-major: core matrix = 8 positions
    // (K) x 8 rows (16 bytes); position groups P_LBO apart, row groups P_SBO apart
    static constexpr int P_LBO = 128, P_SBO = (kVM / 8) * P_LBO, PBUF = (kVN / 8) * P_SBO;
    static constexpr int K_OFF = 0;
    static constexpr int VH_OFF = K_OFF + KBUF;                      // [2 halves]
    static constexpr int VL_OFF = VH_OFF + 2 * VBUF;                 // [2 halves]
    static constexpr int Q_OFF = VL_OFF + 2 * VBUF;
    static constexpr int PH_OFF = Q_OFF + QBUF, PL_OFF = PH_OFF + PBUF;
    static constexpr int RAW_OFF = PL_OFF + PBUF;
    static constexpr int SKF_OFF = RAW_OFF + RS * RAW;               // fp32 [2][block][128 positions]
    static constexpr int SQ_OFF = SKF_OFF + 2 * kNB * kVM * 4;       // fp32 [block][32 rows]
    static constexpr int REC_OFF = SQ_OFF + kNB * kVN * 4;           // int4 [RS][kVSub]
    static constexpr int NSUB_OFF = REC_OFF + RS * kVSub * 16;       // int [RS]
    static constexpr int OREC_OFF = (NSUB_OFF + RS * 4 + 15) / 16 * 16;   // int4 [2][kVSub]
    static constexpr int ONSUB_OFF = OREC_OFF + 2 * kVSub * 16;      // int [2]
    static constexpr int XF_OFF = (ONSUB_OFF + 8 + 15) / 16 * 16;    // int [2 halves][2 parity][4 quarters]
    static constexpr int XM_OFF = XF_OFF + 2 * 2 * 4 * 4;            // fp32 [2 halves][2 parity][16 rows][4 quarters]
    static constexpr int WALK_OFF = XM_OFF + 2 * 2 * 16 * 4 * 4;    // the copy issuer's Walk and stage count
    static constexpr int BAR_OFF = WALK_OFF + (int)((sizeof(Walk) + 4 + 15) / 16 * 16);
    // barriers (arrivals per phase): raw[RS] (copy bytes), k_ready[2] (2 K warps),
    // s_full[2] (commit), s_free[2] (8 softmax warps), v_ready[2 halves] (4 V warps),
    // pv_done[2 halves] (commit), p_ready (8), fin (2 commits), x[2 row halves] (4 warps)
    static constexpr int B_RAW = 0, B_KR = RS, B_SFULL = RS + 2, B_SFREE = RS + 4, B_VR = RS + 6;
    static constexpr int B_PV = RS + 8, B_PREADY = RS + 10, B_FIN = RS + 11, B_X = RS + 12, NBAR = RS + 14;
    static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;              // tmem base, bad flag
    static constexpr int SMEM = MISC_OFF + 16;
    static_assert(RAW % 16 == 0 && R_KS % 16 == 0 && R_V % 16 == 0 && R_VS % 16 == 0, "16-byte granules");
    static_assert(VH_OFF % 16 == 0 && Q_OFF % 16 == 0 && PH_OFF % 16 == 0 && RAW_OFF % 16 == 0, "16-byte operands");
    static_assert(SMEM <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
    static_assert(RAW_OFF < (1 << 18), "operand addresses must fit the descriptor's 18-bit field");
};

// 8 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// Reduce 16 per-lane values over the 32 lanes of a warp (max or sum): after
// five exchange steps, each of which halves the values a lane keeps, lane l
// holds the result of value l >> 1.
template <bool MAX>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane)
{
    float a[8];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float keep = up ? v[k + 8] : v[k], give = up ? v[k] : v[k + 8];
            const float got = __shfl_xor_sync(0xffffffffu, give, 16);
            a[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    float b4[4];
    {
        const bool up = lane & 8;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float keep = up ? a[k + 4] : a[k], give = up ? a[k] : a[k + 4];
            const float got = __shfl_xor_sync(0xffffffffu, give, 8);
            b4[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    float c2[2];
    {
        const bool up = lane & 4;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float keep = up ? b4[k + 2] : b4[k], give = up ? b4[k] : b4[k + 2];
            const float got = __shfl_xor_sync(0xffffffffu, give, 4);
            c2[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    float d;
    {
        const bool up = lane & 2;
        const float keep = up ? c2[1] : c2[0], give = up ? c2[0] : c2[1];
        const float got = __shfl_xor_sync(0xffffffffu, give, 2);
        d = MAX ? fmaxf(keep, got) : keep + got;
    }
    const float got = __shfl_xor_sync(0xffffffffu, d, 1);
    return MAX ? fmaxf(d, got) : d + got;
}

// Instruction descriptor of kind::f16 with B MN-major (transpose bit 16).
__host__ __device__ constexpr uint32_t umma_idesc_f16_bmn(int m, int n)
{
    return umma_idesc_f16(m, n) | (1u << 16);
}

template <int VT>
__global__ void __launch_bounds__(kVThreads, 1) verify_attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = VerifyCfg<VT>;
    constexpr float kSlack = 3.0f;
    constexpr uint32_t kIdQK = umma_idesc_f16(kVM, kVN), kIdPV = umma_idesc_f16_bmn(kD, kVN);
    extern __shared__ __align__(1024) uint8_t smem[];

    // ---- the group, sequence, kv head and split of this CTA (one row tile) ----
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if ((int)blockIdx.x >= p.grp[k].cta0) gi = k;
    const GroupDesc &G = p.grp[gi];
    const int lb = (int)blockIdx.x - G.cta0;
    const int split = lb % G.n_split, h = (lb / G.n_split) % G.n_kv_heads, b = lb / G.n_split / G.n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gb = p.grp_begin[G.head0 + h], gsz = p.grp_begin[G.head0 + h + 1] - gb;
    const int R = min(kVN, gsz * G.t_q);
    if (R <= 0) return;
    const int seg0 = p.seq_seg0[G.seq0 + b], nseg = p.seq_nseg[G.seq0 + b];
    const int lcap = nseg ? min(G.max_len, p.seg[seg0 + nseg - 1].pos0 + p.seg[seg0 + nseg - 1].cap) : 0;

    pdl_wait();
    pdl_trigger();
    const int L = max(0, min(G.seq_lens[b], lcap));
    // the split's positions, cut at the sequence length and, under the causal
    // tail, after the last position the last query token sees
    const int r0 = split * G.chunk;
    int r1 = min(L, r0 + G.chunk);
    if (G.causal) r1 = min(r1, L - G.t_q + (R - 1) / gsz + 1);
    if (r0 >= r1) {   // nothing visible in this split
        if (tid < R) {
            const int i = tid / gsz, hq = p.grp_q[gb + tid % gsz];
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
    // KV tiles: each segment piece of [r0, r1) in runs of up to kVSub cache tiles
    int n_tiles = 0;
    for (int k = 0; k < nseg; ++k) {
        const SegDesc &s = p.seg[seg0 + k];
        const int end = (k + 1 < nseg) ? p.seg[seg0 + k + 1].pos0 : s.pos0 + s.cap;
        const int a = max(r0, s.pos0), e = min(min(r1, end), s.pos0 + s.cap);
        if (a < e) {
            const int n16 = (e - s.pos0 + kWTile - 1) / kWTile - (a - s.pos0) / kWTile;
            n_tiles += (n16 + kVSub - 1) / kVSub;
        }
    }

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::BAR_OFF;
    auto bar = [&](int k) { return bars + 8u * (uint32_t)k; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *bad = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    if (warp == kVKWarp0) tmem_alloc(smem_u32(tmem_slot), 512);
    if (tid == 0) {
        *bad = 0;
        for (int k = 0; k < C::NBAR; ++k) {
            int n = 1;                                                          // raw, s_full, pv_done, fin
            if (k == C::B_KR || k == C::B_KR + 1) n = kVKWarps;
            else if (k == C::B_FIN) n = 2;
            else if (k == C::B_SFREE || k == C::B_SFREE + 1 || k == C::B_PREADY) n = kVSoftWarps;
            else if (k == C::B_VR || k == C::B_VR + 1 || k == C::B_X || k == C::B_X + 1) n = 4;
            mbar_init(bar(k), n);
        }
        fence_mbar_init();
    }

    // ---- the query rows (int8 rule, fp16 scale per 32-block) as exact fp16
    // codes in the Q operand, and their scales: thread u < 128 takes row u / 4,
    // block u % 4 (rows past R are zero) ----
    if (tid < kVN * kNB) {
        const int row = tid >> 2, bb = tid & 3;
        uint32_t wv[16];
        float sc = 0.f;
        if (row < R) {
            const int i = row / gsz, hq = p.grp_q[gb + row % gsz];
            const uint4 *src = reinterpret_cast<const uint4 *>(G.q + (((size_t)b * G.t_q + i) * G.n_q_heads + hq) * kD);
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
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) wv[e] = 0u;
        }
        reinterpret_cast<float *>(smem + C::SQ_OFF)[bb * kVN + row] = sc * G.qk_scale_log2;
        uint8_t *qop = smem + C::Q_OFF + (row / 8) * C::Q_SBO + (row % 8) * 16;
#pragma unroll
        for (int k = 0; k < 4; ++k)   // dims 32bb + 8k .. +7 = core matrix 4bb + k along K
            *reinterpret_cast<uint4 *>(qop + (4 * bb + k) * 128) =
                make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();   // barriers, the TMEM base, the Q operand and the query scales in place
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S_b of tile parity j & 1 at 128 (j & 1) + 32 b (lane =
    // position, column = row), O^T at 256..287 (lane = head dim, column = row)
    const uint32_t tS = tmem, tO = tmem + 256;

    auto give_up = [&]() {
        if (!*bad) {
            *bad = 1;
            atomicAdd(p.timeouts, 1u);
        }
    };
    auto wwait = [&](uint32_t b_, uint32_t parity) {
        const bool okw = mbar_wait(b_, parity);
        return __all_sync(0xffffffffu, okw);
    };
    auto wbad = [&]() { return __any_sync(0xffffffffu, *bad != 0); };

    if (warp >= kVKWarp0) {
        // ================= convert: cache codes -> fp16 operands =================
        const bool kside = warp < kVVWarp0;
        const int kt = tid - 32 * kVKWarp0, ct = tid - 32 * kVVWarp0;
        const bool qk_lane = warp == kVKWarp0 && lane == 0;   // issues the QK MMAs of each tile
        // k16-step descriptors differ from a base only in the start address
        // (16-byte units, no carry out of its 14 bits)
        const uint64_t dK = umma_desc(sbase + C::K_OFF, C::K_LBO, C::K_SBO);
        const uint64_t dQ = umma_desc(sbase + C::Q_OFF, 128, C::Q_SBO);
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            const int st = j % C::RS, ob = j & 1;
            if (!wwait(bar(C::B_RAW + st), (j / C::RS) & 1)) { give_up(); break; }
            const uint8_t *raw = smem + C::RAW_OFF + st * C::RAW;
            const int4 *rec = reinterpret_cast<const int4 *>(smem + C::REC_OFF) + st * kVSub;
            const int ns = reinterpret_cast<const int *>(smem + C::NSUB_OFF)[st];
            // slot k (cache tile k / 16, position k % 16) holds a visible cache
            // row?  One bit per slot, from four ballots of the warp.
            uint32_t vm[4];
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const int k = 32 * hh + lane, t4 = k / kWTile, u = k % kWTile;
                const int4 r = rec[t4];
                vm[hh] = __ballot_sync(0xffffffffu, t4 < ns && r.x + u >= r.y && r.x + u < r.z && r.w + u < L);
            }
            auto slot_ok = [&](int k) { return (vm[k >> 5] >> (k & 31)) & 1u; };
            if (kside) {
                // the K operand is free once QK(j-1) is done; the scale and record
                // slots of parity ob once the softmax has read tile j-2
                if (j >= 1 && !wwait(bar(C::B_SFULL + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { give_up(); break; }
                if (j >= 2 && !wwait(bar(C::B_SFREE + ob), ((j - 2) >> 1) & 1)) { give_up(); break; }
                if (kt < kVSub) reinterpret_cast<int4 *>(smem + C::OREC_OFF)[ob * kVSub + kt] = rec[kt];
                if (kt == 0) reinterpret_cast<int *>(smem + C::ONSUB_OFF)[ob] = ns;
                // K codes: 16-byte chunk ci = 32 i + ln of a cache tile holds
                // position 8 (i / 2) + ln / 4, dims 64 (i % 2) + 8 (ln % 4) + 0..7
                // and the same + 32
                uint8_t *kop = smem + C::K_OFF;
#pragma unroll 4
                for (int mm = 0; mm < kVSub * (C::TILE_K / 16) / (32 * kVKWarps); ++mm) {
                    const int cidx = kt + 32 * kVKWarps * mm;
                    const int t4 = cidx / (C::TILE_K / 16), ci = cidx % (C::TILE_K / 16), i = ci >> 5, ln = ci & 31;
                    const int pos = kWTile * t4 + 8 * (i >> 1) + (ln >> 2);
                    const int dg0 = 8 * (i & 1) + (ln & 3);
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                    if (slot_ok(pos)) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(raw + C::R_K + t4 * C::TILE_K + ci * 16);
                        lo = i8x8_to_f16(w.x, w.y);
                        hi = i8x8_to_f16(w.z, w.w);
                    }
                    *reinterpret_cast<uint4 *>(kop + (pos / 8) * C::K_SBO + dg0 * C::K_LBO + (pos % 8) * 16) = lo;
                    *reinterpret_cast<uint4 *>(kop + (pos / 8) * C::K_SBO + (dg0 + 4) * C::K_LBO + (pos % 8) * 16) = hi;
                }
                // K scales as fp32 [block][position]
                float *skf = reinterpret_cast<float *>(smem + C::SKF_OFF) + ob * kNB * kVM;
#pragma unroll
                for (int e = 0; e < kVM / (32 * kVKWarps); ++e) {
                    const int pos = kt + 32 * kVKWarps * e, t4 = pos / kWTile, u = pos % kWTile;
                    float x[4] = {0.f, 0.f, 0.f, 0.f};
                    if (slot_ok(pos)) load4h(reinterpret_cast<const uint16_t *>(raw + C::R_KS + t4 * C::TILE_S) + u * kNB, x);
#pragma unroll
                    for (int bb = 0; bb < kNB; ++bb) skf[bb * kVM + pos] = x[bb];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_KR + ob));
                if (qk_lane) {
                    // ---- QK MMAs: S_b^T(j) = K_b(j) Q_b^T, once every K warp is
                    // done and the softmax has read S(j-2) ----
                    bool okq = mbar_wait(bar(C::B_KR + ob), (j >> 1) & 1);
                    if (okq && j >= 2) okq = mbar_wait(bar(C::B_SFREE + ob), ((j - 2) >> 1) & 1);
                    if (!okq) {
                        give_up();
                    } else {
                        tc_fence_after();
                        const uint32_t dS = tS + 128 * ob;
#pragma unroll
                        for (int bb = 0; bb < kNB; ++bb)
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const int kc = 4 * bb + 2 * kk;   // first core matrix of the step along K
                                umma_f16(dS + 32 * bb, dK + (uint64_t)(kc * (C::K_LBO / 16)), dQ + (uint64_t)(kc * 8),
                                         kIdQK, kk);
                            }
                        umma_commit(bar(C::B_SFULL + ob));
                    }
                }
                __syncwarp();
            } else {
                // V: v / 2 = code * (d / 2) as fp16 hi + lo, stored [dim][position]
                // in the half's operand once P.V(j-1) of that half is done
                bool ok = true;
                for (int hh = 0; hh < 2; ++hh) {
                    if (j >= 1 && !wwait(bar(C::B_PV + hh), (j - 1) & 1)) { give_up(); ok = false; break; }
                    uint8_t *vh = smem + C::VH_OFF + hh * C::VBUF, *vl = smem + C::VL_OFF + hh * C::VBUF;
                    auto put = [&](int dim, int posl, uint32_t code2, __half2 d2) {
                        uint32_t hi, lo;
                        v_hilo(code2, d2, hi, lo);
                        const int o = (dim / 8) * C::V_SBO + (posl / 8) * 128 + (dim % 8) * 16 + (posl % 8) * 2;
                        *reinterpret_cast<uint32_t *>(vh + o) = hi;
                        *reinterpret_cast<uint32_t *>(vl + o) = lo;
                    };
                    constexpr int CPT = C::TILE_V / 16;                      // 16-byte chunks per cache tile
                    constexpr int NCH = (kVSub / 2) * CPT / 128;             // chunks per converter thread per half
#pragma unroll
                    for (int k = 0; k < NCH; ++k) {
                        const int cidx = ct + 128 * k;
                        const int t4 = (kVSub / 2) * hh + cidx / CPT, ci = cidx % CPT;
                        const int i = ci / 32, ln = ci % 32, g = ln >> 2, c = ln & 3;
                        const uint4 w = *reinterpret_cast<const uint4 *>(raw + C::R_V + t4 * C::TILE_V + ci * 16);
                        const int t = (VT == KVQ_V_Q4_0) ? 8 * i + 2 * c : 8 * (i >> 1) + 2 * c;
                        const int posl = kWTile * (t4 - (kVSub / 2) * hh) + t;   // position in the half
                        // scales of positions t, t + 1 (0 where the slot holds no visible row), times 1/2
                        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                        const uint16_t *vs = reinterpret_cast<const uint16_t *>(raw + C::R_VS + t4 * C::TILE_S);
                        if (slot_ok(kWTile * t4 + t)) load4h(vs + t * kNB, d0);
                        if (slot_ok(kWTile * t4 + t + 1)) load4h(vs + (t + 1) * kNB, d1);
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
                                put(32 * bb + 2 * g, posl, *reinterpret_cast<uint32_t *>(&cv), d2);
                                x = (w23 & 0x000F000Fu) | 0x64006400u;
                                cv = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
                                put(32 * bb + 2 * g + 1, posl, *reinterpret_cast<uint32_t *>(&cv), d2);
                                x = (w0 & 0x00F000F0u) | 0x64006400u;
                                cv = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
                                put(32 * bb + 2 * g + 16, posl, *reinterpret_cast<uint32_t *>(&cv), d2);
                                x = (w23 & 0x00F000F0u) | 0x64006400u;
                                cv = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
                                put(32 * bb + 2 * g + 17, posl, *reinterpret_cast<uint32_t *>(&cv), d2);
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
                                        put(32 * bb + 4 * g + 2 * wd + e, posl, *reinterpret_cast<const uint32_t *>(&cv), d2);
                                    }
                                }
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_VR + hh));
                }
                if (!ok) break;
            }
        }
        if (qk_lane) {
            umma_commit(bar(C::B_FIN));
            if (!mbar_wait(bar(C::B_FIN), 0)) give_up();
        }
        __syncwarp();
    } else {
        // ================= softmax: scores, P, final O =================
        // This thread: position t of each KV tile (TMEM lane t of S) and head
        // dim t of O^T (the same lane), rows 16 hr .. 16 hr + 15 (columns).
        const int qq = warp & 3, hr = warp >> 2;
        const uint32_t lane_base = (uint32_t)(32 * qq) << 16;
        const int t = 32 * qq + lane;
        const float *sq = reinterpret_cast<const float *>(smem + C::SQ_OFF);   // [block][row]
        int *xf = reinterpret_cast<int *>(smem + C::XF_OFF);                  // [hr][parity][quarter]
        float *xm = reinterpret_cast<float *>(smem + C::XM_OFF);              // [hr][parity][row][quarter]
        // last visible position of the half's first live row (rows see more
        // positions as their query token index grows); INT_MAX with no live row
        const int lim_min = (16 * hr < R) ? (G.causal ? L - G.t_q + (16 * hr) / gsz : L - 1) : INT_MAX;
        float m[16], l[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
        }
        int xph = 0;           // phases of this row half's exchange barrier so far
        bool o_live = false;   // O^T holds an earlier tile's P.V
        // ---- warp 0, lane 0: the bulk copies of the tiles RS ahead and the P.V
        // MMAs (O^T += V^T P^T, half by half) of each tile once every softmax
        // warp has written its P ----
        const bool pv_lane = warp == 0 && lane == 0;
        int4 *rec = reinterpret_cast<int4 *>(smem + C::REC_OFF);
        int *nsub = reinterpret_cast<int *>(smem + C::NSUB_OFF);
        // (kept in shared memory: only this lane uses them, and registers are
        // what the softmax threads run short of)
        Walk &w = *reinterpret_cast<Walk *>(smem + C::WALK_OFF);
        int &issued = *reinterpret_cast<int *>(smem + C::WALK_OFF + sizeof(Walk));
        auto issue = [&]() {
            const int st = issued % C::RS;
            const int n = min(kVSub, w.Tend - w.T);
            for (int k = 0; k < kVSub; ++k) {
                const int tb = (w.T + k) * kWTile;
                rec[st * kVSub + k] = make_int4(tb, w.la, w.le, w.pos0 + tb);
            }
            nsub[st] = n;
            const uint32_t dst = sbase + C::RAW_OFF + st * C::RAW, bw = bar(C::B_RAW + st);
            mbar_arrive_expect_tx(bw, n * C::TILE);
            bulk_g2s(dst + C::R_K, w.gk, n * C::TILE_K, bw);
            bulk_g2s(dst + C::R_KS, w.gks, n * C::TILE_S, bw);
            bulk_g2s(dst + C::R_V, w.gv, n * C::TILE_V, bw);
            bulk_g2s(dst + C::R_VS, w.gvs, n * C::TILE_S, bw);
            w.T += n;
            w.gk += n * C::TILE_K;
            w.gks += n * C::TILE_S;
            w.gv += n * C::TILE_V;
            w.gvs += n * C::TILE_S;
            if (w.T >= w.Tend) walk_seek(p, seg0, nseg, h, r0, r1, w.k + 1, C::VCODE, w);
            ++issued;
        };
        if (pv_lane) {
            issued = 0;
            walk_seek(p, seg0, nseg, h, r0, r1, 0, C::VCODE, w);
            while (issued < min(C::RS, n_tiles)) issue();
        }
        __syncwarp();
        auto pv_issue = [&](int j) {
            const uint64_t dPH = umma_desc(sbase + C::PH_OFF, C::P_LBO, C::P_SBO);
            const uint64_t dPL = umma_desc(sbase + C::PL_OFF, C::P_LBO, C::P_SBO);
            if (!mbar_wait(bar(C::B_PREADY), j & 1)) return false;
            for (int hh = 0; hh < 2; ++hh) {
                if (!mbar_wait(bar(C::B_VR + hh), j & 1)) return false;
                tc_fence_after();
                const uint64_t dVH = umma_desc(sbase + C::VH_OFF + hh * C::VBUF, 128, C::V_SBO);
                const uint64_t dVL = umma_desc(sbase + C::VL_OFF + hh * C::VBUF, 128, C::V_SBO);
#pragma unroll
                for (int ks = 0; ks < kVHalf / 16; ++ks) {
                    const uint64_t ov = (uint64_t)(16 * ks);                  // 2 core matrices (256 B) along positions
                    const uint64_t op = (uint64_t)(2 * (4 * hh + ks) * (C::P_LBO / 16));
                    umma_f16(tO, dVH + ov, dPH + op, kIdPV, (j > 0 || hh > 0 || ks > 0) ? 1u : 0u);
                    umma_f16(tO, dVH + ov, dPL + op, kIdPV, 1u);
                    umma_f16(tO, dVL + ov, dPH + op, kIdPV, 1u);
                }
                umma_commit(bar(C::B_PV + hh));
            }
            // both converters are done with tile j's raw stage (the V warps said
            // so; the K warps before QK(j), which every softmax warp passed)
            if (issued < n_tiles) issue();
            return true;
        };
        for (int j = 0; j < n_tiles; ++j) {
            if (wbad()) break;
            const int ob = j & 1;
            if (!wwait(bar(C::B_SFULL + ob), (j >> 1) & 1) || !wwait(bar(C::B_KR + ob), (j >> 1) & 1)) {
                give_up();
                break;
            }
            tc_fence_after();
            float sk[kNB];
            {
                const float *skf = reinterpret_cast<const float *>(smem + C::SKF_OFF) + ob * kNB * kVM;
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) sk[bb] = skf[bb * kVM + t];
            }
            const int4 r4 = reinterpret_cast<const int4 *>(smem + C::OREC_OFF)[ob * kVSub + t / kWTile];
            const int ns = reinterpret_cast<const int *>(smem + C::ONSUB_OFF)[ob];
            const int u = t % kWTile, pos = r4.w + u;
            const bool live = t / kWTile < ns && r4.x + u >= r4.y && r4.x + u < r4.z && pos < L;
            float s[16];
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                uint32_t a[kNB][8];
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) tmem_ld8(tS + lane_base + 128 * ob + 32 * bb + 16 * hr + 8 * c8, a[bb]);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int bb = 0; bb < kNB; ++bb) {
                        const float2 q2 = *reinterpret_cast<const float2 *>(sq + bb * kVN + 16 * hr + 8 * c8 + e);
                        acc = fma2(mul2(make_float2(__uint_as_float(a[bb][e]), __uint_as_float(a[bb][e + 1])),
                                        make_float2(sk[bb], sk[bb])),
                                   q2, acc);
                    }
                    s[8 * c8 + e] = acc.x;
                    s[8 * c8 + e + 1] = acc.y;
                }
            }
            if (!live) {
#pragma unroll
                for (int i = 0; i < 16; ++i) s[i] = -INFINITY;
            } else if (pos > lim_min) {   // the causal tail: rows whose query token does not see pos
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = 16 * hr + i;
                    const int lim = r < R ? (G.causal ? L - G.t_q + r / gsz : L - 1) : INT_MAX;
                    if (pos > lim) s[i] = -INFINITY;
                }
            }
            // S(j), the K scales and the slot records of tile j are read: the
            // next QK and the K converters may go on
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_SFREE + ob));

            // ---- lazy reference max, agreed by the four warps of this row half ----
            bool need = false;
#pragma unroll
            for (int i = 0; i < 16; ++i) need |= s[i] > m[i] + kSlack;
            const bool wneed = __any_sync(0xffffffffu, need);
            int par = xph & 1;
            if (lane == 0) xf[(hr * 2 + par) * 4 + qq] = wneed ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_X + hr));
            if (!wwait(bar(C::B_X + hr), par)) { give_up(); break; }
            ++xph;
            const int4 f4 = *reinterpret_cast<const int4 *>(xf + (hr * 2 + par) * 4);
            const bool any = (f4.x | f4.y | f4.z | f4.w) != 0;
            if (any) {   // the exact tile maximum of every row of the half, then the new references
                float alpha[16];
                const float tmx = warp_reduce16<true>(s, lane);   // row lane / 2 over this warp's positions
                par = xph & 1;
                if (!(lane & 1)) xm[((hr * 2 + par) * 16 + (lane >> 1)) * 4 + qq] = tmx;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_X + hr));
                if (!wwait(bar(C::B_X + hr), par)) { give_up(); break; }
                ++xph;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 v = *reinterpret_cast<const float4 *>(xm + ((hr * 2 + par) * 16 + i) * 4);
                    const float mnew = fmaxf(m[i], fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                    alpha[i] = (m[i] == -INFINITY) ? 0.f : fast_exp2(m[i] - mnew);
                    l[i] *= alpha[i];
                    m[i] = mnew;
                }
                if (o_live) {   // O^T *= alpha on this half's columns (this warp's 32 head dims), once P.V(j-1) is done
                    if (!wwait(bar(C::B_PV + 1), (j - 1) & 1)) { give_up(); break; }
                    tc_fence_after();
                    uint32_t o[16];
                    tmem_ld16(tO + lane_base + 16 * hr, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha[k]);
                    tmem_st16(tO + lane_base + 16 * hr, o);
                    tmem_wait_st();
                }
            }
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float2 mu = make_float2(m[i] == -INFINITY ? 0.f : m[i], m[i + 1] == -INFINITY ? 0.f : m[i + 1]);
                const float2 d = sub2(make_float2(s[i], s[i + 1]), mu);
                s[i] = fast_exp2(d.x);
                s[i + 1] = fast_exp2(d.y);
                l[i] += s[i];
                l[i + 1] += s[i + 1];
            }
            // P(j) may overwrite P(j-1), and O^T is stable, once P.V(j-1) is done
            if (j > 0) {
                if (!wwait(bar(C::B_PV + 1), (j - 1) & 1)) { give_up(); break; }
                tc_fence_after();
            }
            // P hi / lo of position t, rows 16hr + 8c8 .. + 7: one 16-byte row of a
            // core matrix of the MN-major operand
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = make_float2(s[8 * c8 + 2 * e], s[8 * c8 + 2 * e + 1]);
                    const uint32_t hp = pack_half2(x.x, x.y);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hp));
                    const float2 lo = sub2(x, hf);
                    hw[e] = hp;
                    lw[e] = pack_half2(lo.x, lo.y);
                }
                const int off = (2 * hr + c8) * C::P_SBO + (t / 8) * C::P_LBO + (t % 8) * 16;
                *reinterpret_cast<uint4 *>(smem + C::PH_OFF + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(smem + C::PL_OFF + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PREADY));
            o_live = true;
            if (warp == 0) {
                if (pv_lane && !pv_issue(j)) give_up();
                __syncwarp();
            }
        }
        // drain: every P.V MMA, and the copies no converter took
        if (pv_lane) {
            umma_commit(bar(C::B_FIN));
            if (!mbar_wait(bar(C::B_FIN), 0)) give_up();
            for (int k = max(0, issued - C::RS); k < issued; ++k) mbar_wait(bar(C::B_RAW + k % C::RS), (k / C::RS) & 1);
        }
        __syncwarp();
        // ---- final: the rows' sums over the 128 positions of a tile (the four
        // warps of the half), then O^T column by column ----
        bool ok = !wbad();
        float lt[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) lt[i] = 0.f;
        if (ok) {
            ok = wwait(bar(C::B_PV + 1), (n_tiles - 1) & 1);
            tc_fence_after();
            if (ok) {
                const float ls = warp_reduce16<false>(l, lane);
                const int par = xph & 1;
                if (!(lane & 1)) xm[((hr * 2 + par) * 16 + (lane >> 1)) * 4 + qq] = ls;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_X + hr));
                ok = wwait(bar(C::B_X + hr), par);
                if (ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 v = *reinterpret_cast<const float4 *>(xm + ((hr * 2 + par) * 16 + i) * 4);
                        lt[i] = (v.x + v.y) + (v.z + v.w);
                    }
                }
            }
            if (!ok) give_up();
        }
        const bool lost = !ok || wbad();
        uint32_t o[16];
        tmem_ld16(tO + lane_base + 16 * hr, o);   // every lane of the warp takes part
        tmem_wait_ld();
        const float nan = __int_as_float(0x7fc00000);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int r = 16 * hr + k;
            if (r >= R) continue;
            const int i = r / gsz, hq = p.grp_q[gb + r % gsz];
            const size_t orow = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
            float val = nan, lse = nan;
            if (!lost) {
                const bool anyl = lt[k] > 0.f;
                float inv, lg;
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(lt[k]));
                asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(lt[k]));
                val = anyl ? __uint_as_float(o[k]) * (inv / kPVScale) : 0.f;
                lse = anyl ? (m[k] + lg) * 0.69314718055994531f : -INFINITY;
            }
            if (G.n_split == 1) {
                G.out[orow * kD + t] = val;
                if (qq == 0 && lane == k) G.lse[orow] = lse;
            } else {
                G.ws_o[(orow * G.n_split + split) * kD + t] = val;
                if (qq == 0 && lane == k) G.ws_lse[orow * G.n_split + split] = lse;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kVKWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int VT>
cudaError_t launch_verify_t(const AttnParams &p, int n_ctas, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(kVThreads);
    cfg.dynamicSmemBytes = VerifyCfg<VT>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_attn_kernel<VT>, p);
}

template <int VT>
cudaError_t prepare_verify_t()
{
    return cudaFuncSetAttribute(verify_attn_kernel<VT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                VerifyCfg<VT>::SMEM);
}

}  // namespace kvq
