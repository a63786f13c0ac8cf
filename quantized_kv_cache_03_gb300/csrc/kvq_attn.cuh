// kvq_attn.cuh -- split-KV decode attention over the quantized cache (sm_103a).
//
// One CTA = (split s, kv head h, sequence b): it attends the query rows of kv
// head h (t_q query tokens x the query heads mapped to h, at most 32 rows) over
// the positions [s*chunk, (s+1)*chunk) of sequence b and writes either the
// final output (one split) or a partial (normalised o, lse) for the combine.
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
//   * QK^T: fp16 tensor-core MMA m16n8k16 on exact integers -- A = the query
//     codes (rows), B = the K codes of 8 positions entered as 1152 + code (one
//     xor and two byte-permutes per packed word), two MMAs per 32-block into
//     one accumulator that starts at -1152 * (sum of the row's codes in the
//     block).  Every partial sum is an integer below 2^24, so the fp32
//     accumulator ends exactly at the integer block dot I_b (never summed
//     across blocks before scaling).  (GB300's int8 mma.sync issues ~8x slower
//     than the fp16 one, which is why the integer dot runs on the fp16 path.)
//   * score = sum_b I_b * (sq_b * sk_b) * sm_scale*log2(e), masked to -inf
//     outside the sequence / causal range; online softmax in base 2 with the
//     running max only raised when some row's maximum grows.
//   * P.V: fp16 tensor-core MMA m16n8k16 with fp32 accumulation.  The V codes
//     enter as exact small integers in fp16 (binary16 exponent trick: 0x6400|n
//     is 1024+n).  The tile layout puts the same head dims of two adjacent
//     positions side by side, which gives the (position, position) pairs the
//     MMA's k dimension needs without a transpose.  The per-(position, block) scale d rides on the P side:
//     B = p*d split into an fp16 high part and an fp16 low part (two MMAs), so
//     P.V keeps ~22 bits of the fp32 product.
//
// Each warp keeps its own (m, l, acc); the four states are merged through
// shared memory at the end in a fixed order.
#pragma once

#include <type_traits>

#include "kvq_internal.cuh"

namespace kvq {

#ifndef KVQ_STAGES_Q4
#define KVQ_STAGES_Q4 3   // 16-position stages per warp ring (q4_0 V)
#endif
#ifndef KVQ_STAGES_Q8
#define KVQ_STAGES_Q8 3   // (q8_0 V)
#endif



template <int NT, int VT>
struct SplitCfg {
    static constexpr int WARPS = split_warps(NT);
    static constexpr int THREADS = WARPS * 32;
    // the <= 8-row kernels are held to 128 registers per thread (512 threads per SM x 4 CTAs of 4 warps,
    // or one CTA of 16 warps); the others take what they need
    static constexpr int MIN_CTAS = (NT == 1) ? (16 / WARPS > 0 ? 16 / WARPS : 1) : 1;
    static constexpr int MTQ = (NT + 1) / 2;                  // 16-row QK m-tiles
    static constexpr int QROWS = 16 * MTQ;                    // query rows kept in smem
    static_assert(QROWS % WARPS == 0, "every warp quantizes the same number of query rows");
    static constexpr int STAGES = (VT == KVQ_V_Q4_0) ? KVQ_STAGES_Q4 : KVQ_STAGES_Q8;   // ring depth per warp
    static constexpr int VCODE = (VT == KVQ_V_Q4_0) ? kD / 2 : kD;            // V code bytes per position
    // one warp stage: one tile of K codes, K scales, V codes, V scales (cache order)
    static constexpr int K_OFF = 0;
    static constexpr int KS_OFF = K_OFF + kWTile * kD;
    static constexpr int V_OFF = KS_OFF + kWTile * kNB * 2;
    static constexpr int VS_OFF = V_OFF + kWTile * VCODE;
    static constexpr int STAGE = VS_OFF + kWTile * kNB * 2;   // = bytes the four copies land
    static constexpr int RING = STAGES * STAGE;               // per warp
    static constexpr int Q_OFF = WARPS * RING;                // int8 [QROWS][kD]
    static constexpr int QS_OFF = Q_OFF + QROWS * kD;         // fp32 [QROWS][kNB]
    static constexpr int QSUM_OFF = QS_OFF + QROWS * kNB * 4; // int32 [QROWS][kNB]
    static constexpr int ML_OFF = QSUM_OFF + QROWS * kNB * 4; // fp32 m, l [WARPS][8*NT]
    // Per-lane query table, [chunk][lane][4 words] (16-byte chunks, lane-major
    // so a warp's LDS.128 of one chunk is conflict free): the query MMA
    // fragments (for NT == 1 only the a0/a2 words of rows 0..7), the lane's
    // query-row scales [NT][kNB] and the QK accumulator seeds.
    static constexpr int QA_CHUNKS = (NT == 1) ? kNB : MTQ * kNB * 2;
    static constexpr int SQ_CHUNKS = NT;
    static constexpr int CI_CHUNKS = (NT == 1) ? 1 : MTQ * 2;
    static constexpr int QF_CHUNKS = QA_CHUNKS + SQ_CHUNKS + CI_CHUNKS;
    static constexpr int QF_OFF = ML_OFF + 2 * WARPS * 8 * NT * 4;
    static constexpr int TI_OFF = QF_OFF + QF_CHUNKS * 32 * 16;  // int4 tile record [WARPS][STAGES]
    static constexpr int BAR_OFF = TI_OFF + WARPS * STAGES * 16; // uint64 mbarrier [WARPS][STAGES]
    static constexpr int FLAG_OFF = BAR_OFF + WARPS * STAGES * 8;
    static constexpr int SMEM = FLAG_OFF + 16;
    static_assert(8 * NT * kD * 4 <= WARPS * RING, "merge buffer must fit in the stage rings");
    static_assert(STAGE % 16 == 0 && KS_OFF % 16 == 0 && V_OFF % 16 == 0 && VS_OFF % 16 == 0, "16-byte granules");
};

// The pieces of a sequence's segments that fall in [r0, r1), walked in order
// in tiles of kWTile positions (local token index T * kWTile of segment k).
struct Walk {
    int k;            // segment table entry (relative to the sequence's first)
    int T;            // tile index inside the segment
    int la, le;       // local range [la, le) of the current piece
    int pos0;
    const uint8_t *kq, *ks, *vq, *vs;   // kv head h's rows of the current segment
};

__device__ __forceinline__ void walk_seek(const AttnParams &p, int seg0, int nseg, int h, int r0, int r1, int k,
                                          int vcode, Walk &w)
{
    for (w.k = k; w.k < nseg; ++w.k) {
        const SegDesc &s = p.seg[seg0 + w.k];
        const int end = (w.k + 1 < nseg) ? p.seg[seg0 + w.k + 1].pos0 : s.pos0 + s.cap;
        const int a = max(r0, s.pos0), e = min(min(r1, end), s.pos0 + s.cap);
        if (a < e) {
            w.la = a - s.pos0;
            w.le = e - s.pos0;
            w.T = w.la / kWTile;
            w.pos0 = s.pos0;
            const size_t row = (size_t)h * s.cap;
            w.kq = reinterpret_cast<const uint8_t *>(s.kq) + row * kD;
            w.ks = reinterpret_cast<const uint8_t *>(s.ks) + row * kNB * 2;
            w.vq = s.vq + row * vcode;
            w.vs = reinterpret_cast<const uint8_t *>(s.vs) + row * kNB * 2;
            return;
        }
    }
}

__device__ __forceinline__ void walk_next(const AttnParams &p, int seg0, int nseg, int h, int r0, int r1, int vcode,
                                          Walk &w)
{
    ++w.T;
    if (w.T * kWTile >= w.le) walk_seek(p, seg0, nseg, h, r0, r1, w.k + 1, vcode, w);
}

// Lane 0 fills ring slot `dst` (shared address) with the walk's current tile:
// four contiguous bulk copies whose bytes complete on the slot's barrier.
// Positions of the tile outside [la, le) are copied too (they are cache rows
// of the same segment, possibly never written) and masked where they are used.
template <int NT, int VT>
__device__ __forceinline__ void tile_issue(const Walk &w, uint32_t dst, uint32_t bar)
{
    using C = SplitCfg<NT, VT>;
    const size_t tb = (size_t)w.T * kWTile;
    mbar_arrive_expect_tx(bar, C::STAGE);
    bulk_g2s(dst + C::K_OFF, w.kq + tb * kD, kWTile * kD, bar);
    bulk_g2s(dst + C::KS_OFF, w.ks + tb * kNB * 2, kWTile * kNB * 2, bar);
    bulk_g2s(dst + C::V_OFF, w.vq + tb * C::VCODE, kWTile * C::VCODE, bar);
    bulk_g2s(dst + C::VS_OFF, w.vs + tb * kNB * 2, kWTile * kNB * 2, bar);
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

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

template <int NT, int VT, bool DUMP>
__global__ void __launch_bounds__(SplitCfg<NT, VT>::THREADS, SplitCfg<NT, VT>::MIN_CTAS)
    split_attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = SplitCfg<NT, VT>;
    constexpr int kWarps = C::WARPS;
    constexpr int kThreads = C::THREADS;
    constexpr int MTQ = C::MTQ;
    constexpr int S = C::STAGES;
    constexpr float kBias = 1152.0f;                 // K codes enter the MMA as 1152 + code
    extern __shared__ __align__(128) uint8_t smem[];

    // ---- the group, sequence, kv head and split of this CTA ----
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if ((int)blockIdx.x >= p.grp[k].cta0) gi = k;
    const GroupDesc &G = p.grp[gi];
    const int lb = (int)blockIdx.x - G.cta0;
    const int split = lb % G.n_split, h = (lb / G.n_split) % G.n_kv_heads, b = lb / G.n_split / G.n_kv_heads;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int gb = p.grp_begin[G.head0 + h], gsz = p.grp_begin[G.head0 + h + 1] - gb;
    const int R = gsz * G.t_q;
    const int seg0 = p.seq_seg0[G.seq0 + b], nseg = p.seq_nseg[G.seq0 + b];
    const int lcap = nseg ? min(G.max_len, p.seg[seg0 + nseg - 1].pos0 + p.seg[seg0 + nseg - 1].cap) : 0;
    // The split's positions as far as the segment table knows them: the
    // sequence length, read below, can only cut them shorter.  Copies of the
    // range go out before that read returns; positions at or past the length
    // are masked like any other invisible position.
    const int r0 = split * G.chunk, r1c = min(lcap, r0 + G.chunk);

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
            const int i = r / gsz, hq = p.grp_q[gb + r % gsz];
            qraw[k] = *reinterpret_cast<const uint2 *>(G.q + (((size_t)b * G.t_q + i) * G.n_q_heads + hq) * kD + lane * 4);
        }
    }
    // ---- this warp's sub-range and its first copies (before the query prologue) ----
    const int span = (r1c - r0 + kWarps * kWTile - 1) / (kWarps * kWTile) * kWTile;
    const int w0 = min(r1c, r0 + warp * span), w1 = min(r1c, w0 + span);
    int n_tiles = 0;
    if (w0 < w1)
        for (int k = 0; k < nseg; ++k) {
            const SegDesc &s = p.seg[seg0 + k];
            const int end = (k + 1 < nseg) ? p.seg[seg0 + k + 1].pos0 : s.pos0 + s.cap;
            const int a = max(w0, s.pos0) - s.pos0, e = min(min(w1, end), s.pos0 + s.cap) - s.pos0;
            if (a < e) n_tiles += (e - 1) / kWTile - a / kWTile + 1;
        }
    uint8_t *ring = smem + warp * C::RING;
    const uint32_t ring_s = smem_u32(ring);
    const uint32_t bar_s = smem_u32(smem + C::BAR_OFF) + warp * S * 8;
    int4 *tile_rec = reinterpret_cast<int4 *>(smem + C::TI_OFF) + warp * S;
    int *bad_flag = reinterpret_cast<int *>(smem + C::FLAG_OFF);
    if (tid == 0) *bad_flag = 0;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < S; ++st) mbar_init(bar_s + st * 8, 1);
        fence_mbar_init();
    }
    __syncwarp();
    Walk pw;
    walk_seek(p, seg0, nseg, h, w0, w1, 0, C::VCODE, pw);
    int issued = 0;   // tiles handed to the copy engine
    auto issue = [&](int slot) {
        if (lane == 0) {
            const int tb = pw.T * kWTile;
            tile_rec[slot] = make_int4(tb, pw.la, pw.le, pw.pos0 + tb);
            tile_issue<NT, VT>(pw, ring_s + slot * C::STAGE, bar_s + slot * 8);
        }
        walk_next(p, seg0, nseg, h, w0, w1, C::VCODE, pw);
        ++issued;
    };
#pragma unroll
    for (int st = 0; st < S - 1; ++st)
        if (st < n_tiles) issue(st);

    const int L = max(0, min(len_b, lcap));
    const int r1 = min(L, r0 + G.chunk);
    if (r0 >= r1) {                                  // no position in this split
        for (int j = 0; j < issued; ++j) mbar_wait(bar_s + (j % S) * 8, (j / S) & 1);
        if (!DUMP && tid < R) {
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
            const int i = r / gsz, hq = p.grp_q[gb + r % gsz];
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

    // Query A fragments (fp16, exact codes).  Within block bb, k16 step ks, this
    // lane's k slots (2c, 2c+1 | 2c+8, 2c+9) carry head dims
    // 32bb + 8c + 4ks + (0, 1 | 2, 3): the bytes of word 8bb + 2c + ks, the same
    // word the lane reads from K, so q.k is unchanged.  Warp 0 writes them, with
    // the row scales and the accumulator seeds (-1152 * sum of the row's codes
    // in the block), to the per-lane table that every stage reads back.
    uint4 *qf = reinterpret_cast<uint4 *>(smem + C::QF_OFF) + lane;   // chunk k at qf[32 * k]
    if (warp == 0) {
#pragma unroll
        for (int mq = 0; mq < MTQ; ++mq)
#pragma unroll
            for (int bb = 0; bb < kNB; ++bb) {
                uint32_t f[2][4];
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint32_t wa = qw[(16 * mq + g) * (kD / 4) + 8 * bb + 2 * c + ks];
                    const uint32_t wb = qw[(16 * mq + g + 8) * (kD / 4) + 8 * bb + 2 * c + ks];
                    f[ks][0] = q_pair(wa, 0);
                    f[ks][1] = q_pair(wb, 0);
                    f[ks][2] = q_pair(wa, 2);
                    f[ks][3] = q_pair(wb, 2);
                }
                if (NT == 1) {
                    qf[32 * bb] = make_uint4(f[0][0], f[0][2], f[1][0], f[1][2]);
                } else {
                    qf[32 * ((mq * kNB + bb) * 2 + 0)] = make_uint4(f[0][0], f[0][1], f[0][2], f[0][3]);
                    qf[32 * ((mq * kNB + bb) * 2 + 1)] = make_uint4(f[1][0], f[1][1], f[1][2], f[1][3]);
                }
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = 8 * nt + g;
            qf[32 * (C::QA_CHUNKS + nt)] =
                make_uint4(__float_as_uint(qs[row * kNB + 0]), __float_as_uint(qs[row * kNB + 1]),
                           __float_as_uint(qs[row * kNB + 2]), __float_as_uint(qs[row * kNB + 3]));
        }
#pragma unroll
        for (int mq = 0; mq < MTQ; ++mq)
#pragma unroll
            for (int hf = 0; hf < (NT == 1 ? 1 : 2); ++hf) {
                const int row = 16 * mq + 8 * hf + g;
                qf[32 * (C::QA_CHUNKS + C::SQ_CHUNKS + mq * 2 + hf)] =
                    make_uint4(__float_as_uint(-kBias * (float)qsum[row * kNB + 0]),
                               __float_as_uint(-kBias * (float)qsum[row * kNB + 1]),
                               __float_as_uint(-kBias * (float)qsum[row * kNB + 2]),
                               __float_as_uint(-kBias * (float)qsum[row * kNB + 3]));
            }
    }
    __syncthreads();   // query table visible
    float m[NT], l[NT];
    int lim[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int row = 8 * nt + g;
        lim[nt] = (row < R) ? (G.causal ? L - G.t_q + row / gsz : L - 1) : -1;
        m[nt] = -INFINITY;
        l[nt] = 0.f;
    }
    const int lim_min = G.causal ? L - G.t_q : L - 1;   // smallest limit over live rows
    float acc[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[mt][nt][k] = 0.f;

    bool bad = false;   // a stage never arrived (the warp then stops and drains)
    for (int j = 0; j < n_tiles; ++j) {
        const bool landed = mbar_wait(bar_s + (j % S) * 8, (j / S) & 1);
        if (!__all_sync(0xffffffffu, landed)) {
            bad = true;
            break;
        }
        __syncwarp();   // every lane is done with stage j-1, whose slot is refilled next
        if (j + S - 1 < n_tiles) {
            if (lane == 0) fence_proxy_async_smem();
            issue((j + S - 1) % S);
        }

        const uint8_t *st = ring + (j % S) * C::STAGE;
        const int4 rec = tile_rec[j % S];
        const int tb = rec.x, la = rec.y, le = rec.z, pos_base = rec.w;
        // every position of the stage valid and visible to every live row?
        const bool full = tb >= la && tb + kWTile <= le && pos_base + kWTile - 1 <= lim_min;

        auto chunk = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            // ---- S = Q K^T per 32-block (exact integers in fp32), scaled scores ----
            uint32_t qa[MTQ][kNB][2][4];
            float cinit[MTQ][kNB][2], sqf[NT][kNB];
#pragma unroll
            for (int mq = 0; mq < MTQ; ++mq)
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) {
                    if (NT == 1) {
                        const uint4 f = qf[32 * bb];
                        qa[mq][bb][0][0] = f.x; qa[mq][bb][0][2] = f.y;
                        qa[mq][bb][1][0] = f.z; qa[mq][bb][1][2] = f.w;
                        qa[mq][bb][0][1] = qa[mq][bb][0][3] = qa[mq][bb][1][1] = qa[mq][bb][1][3] = 0u;
                    } else {
                        const uint4 f0 = qf[32 * ((mq * kNB + bb) * 2 + 0)];
                        const uint4 f1 = qf[32 * ((mq * kNB + bb) * 2 + 1)];
                        qa[mq][bb][0][0] = f0.x; qa[mq][bb][0][1] = f0.y; qa[mq][bb][0][2] = f0.z; qa[mq][bb][0][3] = f0.w;
                        qa[mq][bb][1][0] = f1.x; qa[mq][bb][1][1] = f1.y; qa[mq][bb][1][2] = f1.z; qa[mq][bb][1][3] = f1.w;
                    }
                }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint4 f = qf[32 * (C::QA_CHUNKS + nt)];
                sqf[nt][0] = __uint_as_float(f.x); sqf[nt][1] = __uint_as_float(f.y);
                sqf[nt][2] = __uint_as_float(f.z); sqf[nt][3] = __uint_as_float(f.w);
            }
#pragma unroll
            for (int mq = 0; mq < MTQ; ++mq)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    if (NT == 1 && hf == 1) {
#pragma unroll
                        for (int bb = 0; bb < kNB; ++bb) cinit[mq][bb][1] = 0.f;
                    } else {
                        const uint4 f = qf[32 * (C::QA_CHUNKS + C::SQ_CHUNKS + mq * 2 + hf)];
                        cinit[mq][0][hf] = __uint_as_float(f.x); cinit[mq][1][hf] = __uint_as_float(f.y);
                        cinit[mq][2][hf] = __uint_as_float(f.z); cinit[mq][3][hf] = __uint_as_float(f.w);
                    }
                }
            float s[2][NT][2];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                // K column 8sub + g: load 2sub + hb holds its codes 8c..8c+7 of
                // blocks 2hb and 2hb + 1
                uint4 kk[2];
#pragma unroll
                for (int hb = 0; hb < 2; ++hb)
                    kk[hb] = *reinterpret_cast<const uint4 *>(st + C::K_OFF + (2 * sub + hb) * 512 + lane * 16);
                float sc[MTQ][kNB][4];
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) {
                    const uint32_t kx = (bb & 1) ? kk[bb >> 1].z : kk[bb >> 1].x;
                    const uint32_t ky = (bb & 1) ? kk[bb >> 1].w : kk[bb >> 1].y;
                    uint32_t b00, b01, b10, b11;
                    k_word_biased(kx, b00, b01);
                    k_word_biased(ky, b10, b11);
#pragma unroll
                    for (int mq = 0; mq < MTQ; ++mq) {
                        mma_f16_16816_c(sc[mq][bb], qa[mq][bb][0], b00, b01, cinit[mq][bb][0], cinit[mq][bb][1]);
                        mma_f16_16816(sc[mq][bb], qa[mq][bb][1], b10, b11);
                    }
                }
                // K scales of this lane's two score columns (positions 8sub + 2c + e)
                const int ut = 8 * sub + 2 * c;
                const uint4 ksr = *reinterpret_cast<const uint4 *>(st + C::KS_OFF + ut * kNB * 2);
                float sk[2][kNB];
                {
                    const float2 a0 = __half22float2(*reinterpret_cast<const __half2 *>(&ksr.x));
                    const float2 a1 = __half22float2(*reinterpret_cast<const __half2 *>(&ksr.y));
                    const float2 a2 = __half22float2(*reinterpret_cast<const __half2 *>(&ksr.z));
                    const float2 a3 = __half22float2(*reinterpret_cast<const __half2 *>(&ksr.w));
                    sk[0][0] = a0.x; sk[0][1] = a0.y; sk[0][2] = a1.x; sk[0][3] = a1.y;
                    sk[1][0] = a2.x; sk[1][1] = a2.y; sk[1][2] = a3.x; sk[1][3] = a3.y;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int mq = nt >> 1, idx = 2 * (nt & 1) + e;
                        float a = 0.f;
#pragma unroll
                        for (int bb = 0; bb < kNB; ++bb) a = fmaf(sc[mq][bb][idx], sqf[nt][bb] * sk[e][bb], a);
                        if (FULL) {
                            s[sub][nt][e] = a;
                        } else {
                            const int tok = tb + ut + e;
                            const bool ok = tok >= la && tok < le && pos_base + ut + e <= lim[nt];
                            s[sub][nt][e] = ok ? a : -INFINITY;
                        }
                    }
                if (DUMP) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int row = 8 * nt + g, tok = tb + ut + e, pos = pos_base + ut + e;
                            if (row < R && tok >= la && tok < le && pos < L) {
                                const int mq = nt >> 1, idx = 2 * (nt & 1) + e;
                                const int i = row / gsz, hq = p.grp_q[gb + row % gsz];
                                const size_t o = ((((size_t)b * G.t_q + i) * G.n_q_heads + hq) * G.max_len + pos) * kNB;
                                int4 v;
                                v.x = (int)sc[mq][0][idx]; v.y = (int)sc[mq][1][idx];
                                v.z = (int)sc[mq][2][idx]; v.w = (int)sc[mq][3][idx];
                                *reinterpret_cast<int4 *>(G.dbg_scores + o) = v;
                            }
                        }
                }
            }
            if (DUMP) return;

            // ---- online softmax (base 2) ----
            bool grow = false;
            float mnew[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx = fmaxf(fmaxf(s[0][nt][0], s[0][nt][1]), fmaxf(s[1][nt][0], s[1][nt][1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mnew[nt] = fmaxf(m[nt], mx);
                grow |= mnew[nt] > m[nt];
            }
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float al = (mnew[nt] == -INFINITY) ? 1.f : fast_exp2(m[nt] - mnew[nt]);
                    l[nt] *= al;
                    m[nt] = mnew[nt];
                    const float a0 = __shfl_sync(0xffffffffu, al, 8 * c);       // row 8nt + 2c
                    const float a1 = __shfl_sync(0xffffffffu, al, 8 * c + 4);   // row 8nt + 2c + 1
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        acc[mt][nt][0] *= a0; acc[mt][nt][1] *= a1;
                        acc[mt][nt][2] *= a0; acc[mt][nt][3] *= a1;
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float mu = (m[nt] == -INFINITY) ? 0.f : m[nt];
#pragma unroll
                for (int sub = 0; sub < 2; ++sub)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[sub][nt][e] = fast_exp2(s[sub][nt][e] - mu);
                        l[nt] += s[sub][nt][e];
                    }
            }

            // ---- O += P . V  (per 32-block: B = p*d as fp16 hi + lo, A = V codes) ----
            uint4 vsr[2];   // V scales of this lane's B columns (positions 8sub + 2c, +1)
            bool okv[2][2];
            // V code words of positions (8sub + 2c, +1): q4_0 one load per sub
            // (word bb = block bb), q8_0 two (load 2sub + hb: blocks 2hb, 2hb + 1)
            constexpr int NVL = (VT == KVQ_V_Q4_0) ? 1 : 2;
            uint4 vv[2][NVL];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int ut = 8 * sub + 2 * c;
                vsr[sub] = *reinterpret_cast<const uint4 *>(st + C::VS_OFF + ut * kNB * 2);
                okv[sub][0] = FULL || (tb + ut >= la && tb + ut < le && pos_base + ut < L);
                okv[sub][1] = FULL || (tb + ut + 1 >= la && tb + ut + 1 < le && pos_base + ut + 1 < L);
#pragma unroll
                for (int hb = 0; hb < NVL; ++hb)
                    vv[sub][hb] = *reinterpret_cast<const uint4 *>(st + C::V_OFF + (NVL * sub + hb) * 512 + lane * 16);
            }
#pragma unroll
            for (int bb = 0; bb < kNB; ++bb) {
                uint32_t bhi[NT][2], blo[NT][2];
                uint32_t a[2][4];   // [h2] A fragment of m-tile 2bb + h2
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    // V scale of block bb for the two positions (fp16 -> fp32), 0 if invalid
                    const uint32_t w0 = (bb < 2) ? vsr[sub].x : vsr[sub].y;
                    const uint32_t w1 = (bb < 2) ? vsr[sub].z : vsr[sub].w;
                    float d0 = __half2float(__ushort_as_half((uint16_t)((bb & 1) ? (w0 >> 16) : (w0 & 0xffffu))));
                    float d1 = __half2float(__ushort_as_half((uint16_t)((bb & 1) ? (w1 >> 16) : (w1 & 0xffffu))));
                    if (!FULL) {
                        d0 = okv[sub][0] ? d0 : 0.f;
                        d1 = okv[sub][1] ? d1 : 0.f;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        // x = p*d split as hi (x with its low 13 mantissa bits cleared:
                        // exact in fp16 when x is in fp16's normal range) + lo (x - hi,
                        // exact in fp32, then rounded to fp16)
                        const float x0 = s[sub][nt][0] * d0;
                        const float x1 = s[sub][nt][1] * d1;
                        const float h0 = __uint_as_float(__float_as_uint(x0) & 0xffffe000u);
                        const float h1 = __uint_as_float(__float_as_uint(x1) & 0xffffe000u);
                        bhi[nt][sub] = pack_half2(h0, h1);
                        blo[nt][sub] = pack_half2(x0 - h0, x1 - h1);
                    }
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
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16_16816(acc[2 * bb + h2][nt], a[h2], bhi[nt][0], bhi[nt][1]);
                        mma_f16_16816(acc[2 * bb + h2][nt], a[h2], blo[nt][0], blo[nt][1]);
                    }
            }
        };
        if (full)
            chunk(std::integral_constant<bool, true>());
        else
            chunk(std::integral_constant<bool, false>());
    }

    if (bad) {
        // a wait gave up: wait (bounded) for this warp's copies still in flight,
        // then poison the CTA's results
        for (int j = issued - (S - 1) > 0 ? issued - (S - 1) : 0; j < issued; ++j)
            mbar_wait(bar_s + (j % S) * 8, (j / S) & 1);
        if (lane == 0) {
            atomicOr(bad_flag, 1);
            atomicAdd(p.timeouts, 1u);
        }
    }
    if constexpr (!DUMP) {
        // ---- merge the four warps' (m, l, acc) and write ----
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            l[nt] += __shfl_xor_sync(0xffffffffu, l[nt], 1);
            l[nt] += __shfl_xor_sync(0xffffffffu, l[nt], 2);
        }
        __syncthreads();   // every warp is done with the stage rings
        float *sm_m = reinterpret_cast<float *>(smem + C::ML_OFF);
        float *sm_l = sm_m + kWarps * 8 * NT;
        float *sm_o = reinterpret_cast<float *>(smem);   // [8*NT][kD]
        if (c == 0)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sm_m[warp * 8 * NT + 8 * nt + g] = m[nt];
                sm_l[warp * 8 * NT + 8 * nt + g] = l[nt];
            }
        __syncthreads();
        // Merge in a fixed order so results do not depend on scheduling.  Each
        // (row, dim) belongs to one lane per warp; a warp's accumulator is
        // scaled by exp2(m_warp - M) for the row's overall max M.
        constexpr bool kSlices = kWarps * 8 * NT * kD * 4 <= kWarps * C::RING;
        auto put = [&](float *dst, bool add) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = 8 * nt + 2 * c + e;
                    if (row >= R) continue;
                    float M = -INFINITY;
#pragma unroll
                    for (int v = 0; v < kWarps; ++v) M = fmaxf(M, sm_m[v * 8 * NT + row]);
                    const float mw = sm_m[warp * 8 * NT + row];
                    const float f = (mw == -INFINITY) ? 0.f : fast_exp2(mw - M);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        float *o0 = &dst[row * kD + pv_dim<VT>(mt, g)];
                        float *o1 = &dst[row * kD + pv_dim<VT>(mt, g + 8)];
                        *o0 = (add ? *o0 : 0.f) + acc[mt][nt][e] * f;
                        *o1 = (add ? *o1 : 0.f) + acc[mt][nt][2 + e] * f;
                    }
                }
        };
        if (kSlices) {
            // every warp writes its own slice, then the slices are added 0..3
            put(sm_o + warp * 8 * NT * kD, false);
            __syncthreads();
            for (int i = tid; i < R * kD; i += kThreads) {
                float t = sm_o[i];
#pragma unroll
                for (int w = 1; w < kWarps; ++w) t += sm_o[w * 8 * NT * kD + i];
                sm_o[i] = t;
            }
            __syncthreads();
        } else {
            // warp 0 stores, warps 1..3 add in turn
            for (int w = 0; w < kWarps; ++w) {
                if (warp == w) put(sm_o, w > 0);
                __syncthreads();
            }
        }
        const bool poisoned = *bad_flag != 0;   // set before the merge's first barrier
        for (int i0 = tid; i0 < R * kD; i0 += kThreads) {
            const int row = i0 / kD, d = i0 % kD;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 * NT + row]);
            float Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float mw = sm_m[w * 8 * NT + row];
                if (mw != -INFINITY) Lsum += sm_l[w * 8 * NT + row] * fast_exp2(mw - M);
            }
            const int i = row / gsz, hq = p.grp_q[gb + row % gsz];
            const size_t orow = ((size_t)b * G.t_q + i) * G.n_q_heads + hq;
            const bool any = Lsum > 0.f;
            float inv, lg;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(Lsum));
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(Lsum));
            float o = any ? sm_o[row * kD + d] * inv : 0.f;
            float ls = any ? (M + lg) * 0.69314718055994531f : -INFINITY;
            if (poisoned) o = ls = __int_as_float(0x7fc00000);   // NaN: the CTA lost a stage
            if (G.n_split == 1) {
                G.out[orow * kD + d] = o;
                if (d == 0) G.lse[orow] = ls;
            } else {
                G.ws_o[(orow * G.n_split + split) * kD + d] = o;
                if (d == 0) G.ws_lse[orow * G.n_split + split] = ls;
            }
        }
    }
}

template <int NT, int VT>
cudaError_t launch_split_t(const AttnParams &p, int n_ctas, bool dump, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_ctas);
    cfg.blockDim = dim3(SplitCfg<NT, VT>::THREADS);
    cfg.dynamicSmemBytes = SplitCfg<NT, VT>::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (dump) return cudaLaunchKernelEx(&cfg, split_attn_kernel<NT, VT, true>, p);
    return cudaLaunchKernelEx(&cfg, split_attn_kernel<NT, VT, false>, p);
}

template <int NT, int VT>
cudaError_t prepare_split_t(bool dump, int *ctas_per_sm)
{
    const int smem = SplitCfg<NT, VT>::SMEM;
    const void *fn = dump ? (const void *)split_attn_kernel<NT, VT, true> : (const void *)split_attn_kernel<NT, VT, false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (ctas_per_sm)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, SplitCfg<NT, VT>::THREADS, smem);
    return cudaSuccess;
}

#define KVQ_DEFINE_SPLIT_ENTRY(SUFFIX, VT)                                                   \
    cudaError_t launch_split_##SUFFIX(const AttnParams &p, int nt, int n_ctas, bool dump, cudaStream_t s, bool pdl) \
    {                                                                                        \
        switch (nt) {                                                                        \
        case 1: return launch_split_t<1, VT>(p, n_ctas, dump, s, pdl);                       \
        case 2: return launch_split_t<2, VT>(p, n_ctas, dump, s, pdl);                       \
        case 4: return launch_split_t<4, VT>(p, n_ctas, dump, s, pdl);                       \
        default: return cudaErrorInvalidValue;                                               \
        }                                                                                    \
    }                                                                                        \
    cudaError_t prepare_split_##SUFFIX(int nt, bool dump, int *ctas)                         \
    {                                                                                        \
        switch (nt) {                                                                        \
        case 1: return prepare_split_t<1, VT>(dump, ctas);                                   \
        case 2: return prepare_split_t<2, VT>(dump, ctas);                                   \
        case 4: return prepare_split_t<4, VT>(dump, ctas);                                   \
        default: return cudaErrorInvalidValue;                                               \
        }                                                                                    \
    }

}  // namespace kvq
