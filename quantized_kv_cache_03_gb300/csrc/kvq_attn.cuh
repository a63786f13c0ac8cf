// kvq_attn.cuh -- split-KV decode attention over the quantized cache (sm_103a).
//
// One CTA = (split s, kv head h, sequence b): it attends the query rows of kv
// head h (t_q query tokens x the query heads mapped to h, at most 32 rows) over
// the positions [s*chunk, (s+1)*chunk) of sequence b and writes either the
// final output (one split) or a partial (normalised o, lse) for the combine.
//
// Data path per 64-token stage (cp.async 16-byte copies into a 4-deep shared
// ring, XOR-swizzled so every fragment read below is bank-conflict free):
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
//     enter as exact small integers in fp16 (built from the nibbles/bytes with
//     the binary16 exponent trick: 0x6400|n is 1024+n), turned token-paired by
//     an in-register 8x8 transpose (movmatrix).  The per-(position, block)
//     scale d rides on the P side: B = p*d split into an fp16 high part and an
//     fp16 low part (two MMAs), so P.V keeps ~22 bits of the fp32 product.
//
// Warps: 4, each owns 16 positions of every stage and keeps its own (m, l, acc);
// the four states are merged through shared memory at the end.
#pragma once

#include <type_traits>

#include "kvq_internal.cuh"

namespace kvq {

template <int NT, int VT>
struct SplitCfg {
    static constexpr int MTQ = (NT + 1) / 2;                 // 16-row QK m-tiles
    static constexpr int QROWS = 16 * MTQ;                   // query rows kept in smem
    static constexpr int VROW = (VT == KVQ_V_Q4_0) ? kD / 2 : kD;
    static constexpr int K_OFF = 0;
    static constexpr int KS_OFF = K_OFF + kTile * kD;
    static constexpr int V_OFF = KS_OFF + kTile * kNB * 2;
    static constexpr int VS_OFF = V_OFF + kTile * VROW;
    static constexpr int STAGE = VS_OFF + kTile * kNB * 2;
    static constexpr int Q_OFF = kStages * STAGE;            // int8 [QROWS][kD]
    static constexpr int QS_OFF = Q_OFF + QROWS * kD;        // fp32 [QROWS][kNB]
    static constexpr int QSUM_OFF = QS_OFF + QROWS * kNB * 4; // int32 [QROWS][kNB]
    static constexpr int ML_OFF = QSUM_OFF + QROWS * kNB * 4; // fp32 m, l [kWarps][8*NT]
    static constexpr int SMEM = ML_OFF + 2 * kWarps * 8 * NT * 4;
    static_assert(8 * NT * kD * 4 <= kStages * STAGE, "merge buffer must fit in the stage ring");
};

// Range of segment k of the sequence intersected with [r0, r1): local token
// indices [la, le).  Returns false when empty.
__device__ __forceinline__ bool seg_range(const AttnParams &p, int seg0, int nseg, int k, int r0, int r1,
                                          int &la, int &le)
{
    const SegDesc &s = p.seg[seg0 + k];
    const int end = (k + 1 < nseg) ? p.seg[seg0 + k + 1].pos0 : s.pos0 + s.cap;
    const int a = max(r0, s.pos0);
    const int e = min(min(r1, end), s.pos0 + s.cap);
    la = a - s.pos0;
    le = e - s.pos0;
    return a < e;
}

struct TileCursor {
    int k, T, la, le;
};

__device__ __forceinline__ void cursor_seek(const AttnParams &p, int seg0, int nseg, int r0, int r1,
                                            TileCursor &cur, int from_k)
{
    for (cur.k = from_k; cur.k < nseg; ++cur.k)
        if (seg_range(p, seg0, nseg, cur.k, r0, r1, cur.la, cur.le)) {
            cur.T = cur.la / kTile;
            return;
        }
}

__device__ __forceinline__ void cursor_next(const AttnParams &p, int seg0, int nseg, int r0, int r1,
                                            TileCursor &cur)
{
    ++cur.T;
    if (cur.T * kTile >= cur.le) cursor_seek(p, seg0, nseg, r0, r1, cur, cur.k + 1);
}

// Copy one 64-token stage (K codes, K scales, V codes, V scales of kv head h)
// into shared memory.  Tokens outside [la, le) are zero-filled without a read.
template <int NT, int VT>
__device__ __forceinline__ void issue_stage(const AttnParams &p, const SegDesc &s, int h, const TileCursor &cur,
                                            uint8_t *st, int tid)
{
    using C = SplitCfg<NT, VT>;
    const int tb = cur.T * kTile;
    const size_t hb = (size_t)h * s.cap + tb;   // row of the stage's token 0
#pragma unroll
    for (int i = 0; i < 4; ++i) {               // K: 64 tokens x 8 granules
        const int gi = tid + i * kThreads, u = gi >> 3, part = gi & 7;
        const bool ok = tb + u >= cur.la && tb + u < cur.le;
        const uint32_t *src = s.kq + (hb + u) * (kD / 4) + part * 4;
        cp_async16(smem_u32(st + C::K_OFF + u * kD + ((part ^ (u & 7)) << 4)), ok ? src : s.kq, ok ? 16 : 0);
    }
    if (VT == KVQ_V_Q4_0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {           // V q4_0: 64 tokens x 4 granules
            const int gi = tid + i * kThreads, u = gi >> 2, part = gi & 3;
            const bool ok = tb + u >= cur.la && tb + u < cur.le;
            const uint8_t *src = s.vq + (hb + u) * (kD / 2) + part * 16;
            cp_async16(smem_u32(st + C::V_OFF + u * (kD / 2) + ((part ^ ((u >> 1) & 3)) << 4)),
                       ok ? src : s.vq, ok ? 16 : 0);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {           // V q8_0: 64 tokens x 8 granules
            const int gi = tid + i * kThreads, u = gi >> 3, part = gi & 7;
            const bool ok = tb + u >= cur.la && tb + u < cur.le;
            const uint8_t *src = s.vq + (hb + u) * kD + part * 16;
            cp_async16(smem_u32(st + C::V_OFF + u * kD + ((part ^ (u & 7)) << 4)), ok ? src : s.vq,
                       ok ? 16 : 0);
        }
    }
    if (tid < 64) {                             // scales: 16 B = 2 tokens x 4 blocks
        const int u = 2 * (tid & 31);
        const bool ok = tb + u + 1 >= cur.la && tb + u < cur.le;
        const uint16_t *base = (tid < 32) ? s.ks : s.vs;
        const int off = ((tid < 32) ? C::KS_OFF : C::VS_OFF) + u * kNB * 2;
        cp_async16(smem_u32(st + off), ok ? base + (hb + u) * kNB : base, ok ? 16 : 0);
    }
}

// Head-dim index of accumulator row rho (0..15) of PV m-tile mt = 2*block + h2.
template <int VT>
__device__ __forceinline__ int pv_dim(int mt, int rho)
{
    const int bb = mt >> 1, h2 = mt & 1, gg = rho & 7, half = rho >> 3;
    if (VT == KVQ_V_Q4_0) return 32 * bb + 16 * h2 + 4 * (gg >> 1) + 2 * half + (gg & 1);
    return 32 * bb + 8 * (gg >> 1) + 4 * h2 + 2 * half + (gg & 1);
}

// fp16 pair (elements of two adjacent head dims) -> exact integer values.
template <int VT>
__device__ __forceinline__ void v_codes_to_half2(const uint8_t *st_v, int u, int bb, int c, uint32_t (&P)[4])
{
    if (VT == KVQ_V_Q4_0) {
        // word c of block bb: bytes 4c..4c+3; low nibbles are dims 4c..4c+3,
        // high nibbles dims 16+4c..16+4c+3
        const uint32_t w = *reinterpret_cast<const uint32_t *>(st_v + u * (kD / 2) + ((bb ^ ((u >> 1) & 3)) << 4) +
                                                                4 * c);
        const uint32_t t01 = __byte_perm(w, 0, 0x4140), t23 = __byte_perm(w, 0, 0x4342);
        const __half2 k1032 = __half2half2(__ushort_as_half(0x6408));   // 1032
        const __half2 k16th = __half2half2(__ushort_as_half(0x2c00));   // 1/16
        const __half2 km72 = __half2half2(__ushort_as_half(0xd480));    // -72
        uint32_t x;
        x = (t01 & 0x000F000Fu) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&P[0]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
        x = (t23 & 0x000F000Fu) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&P[1]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1032);
        x = (t01 & 0x00F000F0u) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&P[2]) = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
        x = (t23 & 0x00F000F0u) | 0x64006400u;
        *reinterpret_cast<__half2 *>(&P[3]) = __hfma2(*reinterpret_cast<__half2 *>(&x), k16th, km72);
    } else {
        // words 2c, 2c+1 of block bb: dims 8c..8c+7 as signed bytes
        const uint2 w = *reinterpret_cast<const uint2 *>(st_v + u * kD + (((2 * bb + (c >> 1)) ^ (u & 7)) << 4) +
                                                         ((c & 1) << 3));
        const uint32_t x0 = w.x ^ 0x80808080u, x1 = w.y ^ 0x80808080u;   // biased: code + 128
        const __half2 k1152 = __half2half2(__ushort_as_half(0x6480));     // 1152
        uint32_t x;
        x = __byte_perm(x0, 0x64646464u, 0x4140);
        *reinterpret_cast<__half2 *>(&P[0]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x0, 0x64646464u, 0x4342);
        *reinterpret_cast<__half2 *>(&P[1]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x1, 0x64646464u, 0x4140);
        *reinterpret_cast<__half2 *>(&P[2]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
        x = __byte_perm(x1, 0x64646464u, 0x4342);
        *reinterpret_cast<__half2 *>(&P[3]) = __hsub2(*reinterpret_cast<__half2 *>(&x), k1152);
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

// Two signed int8 codes (bytes k0, k1 of w) -> exact fp16 pair.
__device__ __forceinline__ uint32_t q_pair(uint32_t w, int k0)
{
    const __half2 h = __halves2half2(__int2half_rn((int)(int8_t)(w >> (8 * k0))),
                                     __int2half_rn((int)(int8_t)(w >> (8 * k0 + 8))));
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int NT, int VT, bool DUMP>
__global__ void __launch_bounds__(kThreads) split_attn_kernel(const __grid_constant__ AttnParams p)
{
    using C = SplitCfg<NT, VT>;
    constexpr int MTQ = C::MTQ;
    constexpr float kBias = 1152.0f;                 // K codes enter the MMA as 1152 + code
    extern __shared__ __align__(128) uint8_t smem[];

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
    const int gb = p.grp_begin[h], gsz = p.grp_begin[h + 1] - gb;
    const int R = gsz * p.t_q;
    const int seg0 = p.seq_seg0[b], nseg = p.seq_nseg[b];
    const int lcap = nseg ? min(p.max_len, p.seg[seg0 + nseg - 1].pos0 + p.seg[seg0 + nseg - 1].cap) : 0;

    // Nothing above reads memory written by an earlier kernel.
    pdl_wait();
    pdl_trigger();

    const int L = max(0, min(p.seq_lens[b], lcap));
    const int r0 = split * p.chunk, r1 = min(L, r0 + p.chunk);

    if (r0 >= r1) {                                  // no position in this split
        if (!DUMP && tid < R) {
            const int i = tid / gsz, hq = p.grp_q[gb + tid % gsz];
            const size_t row = ((size_t)b * p.t_q + i) * p.n_q_heads + hq;
            if (p.n_split == 1) {
                p.lse[row] = -INFINITY;
                for (int d = 0; d < kD; ++d) p.out[row * kD + d] = 0.f;
            } else {
                p.ws_lse[row * p.n_split + split] = -INFINITY;
            }
        }
        return;
    }

    // ---- tile schedule; start the copies before the query prologue ----
    int n_tiles = 0;
    for (int k = 0; k < nseg; ++k) {
        int la, le;
        if (seg_range(p, seg0, nseg, k, r0, r1, la, le)) n_tiles += (le - 1) / kTile - la / kTile + 1;
    }
    TileCursor pc, cc;
    cursor_seek(p, seg0, nseg, r0, r1, pc, 0);
    cc = pc;
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
        if (st < n_tiles) {
            issue_stage<NT, VT>(p, p.seg[seg0 + pc.k], h, pc, smem + st * C::STAGE, tid);
            cursor_next(p, seg0, nseg, r0, r1, pc);
        }
        cp_async_commit();
    }

    // ---- quantize the query rows of this kv head (int8 rule, fp16 scale) ----
    uint32_t *qw = reinterpret_cast<uint32_t *>(smem + C::Q_OFF);
    float *qs = reinterpret_cast<float *>(smem + C::QS_OFF);
    int *qsum = reinterpret_cast<int *>(smem + C::QSUM_OFF);
    for (int r = warp; r < C::QROWS; r += kWarps) {
        uint32_t word = 0;
        float s = 0.f;
        int sum = 0;
        if (r < R) {
            const int i = r / gsz, hq = p.grp_q[gb + r % gsz];
            const size_t qrow = ((size_t)b * p.t_q + i) * p.n_q_heads + hq;
            float x[4];
            unpack4h(*reinterpret_cast<const uint2 *>(p.q + qrow * kD + lane * 4), x);
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
                reinterpret_cast<uint32_t *>(p.dbg_qc)[qrow * (kD / 4) + lane] = word;
                if ((lane & 7) == 0) p.dbg_qs[qrow * kNB + (lane >> 3)] = __half_as_ushort(sh);
            }
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        qw[r * (kD / 4) + lane] = word;
        if ((lane & 7) == 0) {
            qs[r * kNB + (lane >> 3)] = s * p.qk_scale_log2;
            qsum[r * kNB + (lane >> 3)] = sum;
        }
    }
    __syncthreads();   // query codes visible

    // Query A fragments (fp16, exact codes).  Within block bb, k16 step ks, this
    // lane's k slots (2c, 2c+1 | 2c+8, 2c+9) carry head dims
    // 32bb + 8c + 4ks + (0, 1 | 2, 3): the bytes of word 8bb + 2c + ks, the same
    // word the lane reads from K, so q.k is unchanged.
    uint32_t qa[MTQ][kNB][2][4];
    float cinit[MTQ][kNB][2];   // -1152 * sum of the row's codes in the block
#pragma unroll
    for (int mq = 0; mq < MTQ; ++mq)
#pragma unroll
        for (int bb = 0; bb < kNB; ++bb) {
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint32_t w0 = qw[(16 * mq + g) * (kD / 4) + 8 * bb + 2 * c + ks];
                const uint32_t w1 = qw[(16 * mq + g + 8) * (kD / 4) + 8 * bb + 2 * c + ks];
                qa[mq][bb][ks][0] = q_pair(w0, 0);
                qa[mq][bb][ks][2] = q_pair(w0, 2);
                // with at most 8 rows, rows 8..15 of the tile are padding: keep them
                // compile-time zeros so they occupy no registers
                qa[mq][bb][ks][1] = NT == 1 ? 0u : q_pair(w1, 0);
                qa[mq][bb][ks][3] = NT == 1 ? 0u : q_pair(w1, 2);
            }
            cinit[mq][bb][0] = -kBias * (float)qsum[(16 * mq + g) * kNB + bb];
            cinit[mq][bb][1] = NT == 1 ? 0.f : -kBias * (float)qsum[(16 * mq + g + 8) * kNB + bb];
        }
    float sqf[NT][kNB], m[NT], l[NT];
    int lim[NT];
    int lim_min = 0x7fffffff;   // smallest visible-position limit over live rows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int row = 8 * nt + g;
#pragma unroll
        for (int bb = 0; bb < kNB; ++bb) sqf[nt][bb] = qs[row * kNB + bb];
        lim[nt] = (row < R) ? (p.causal ? L - p.t_q + row / gsz : L - 1) : -1;
        m[nt] = -INFINITY;
        l[nt] = 0.f;
    }
    lim_min = p.causal ? L - p.t_q : L - 1;
    float acc[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[mt][nt][k] = 0.f;

    const int u0w = warp * 16;   // this warp's first token of every stage

    for (int j = 0; j < n_tiles; ++j) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        if (j + kStages - 1 < n_tiles) {
            issue_stage<NT, VT>(p, p.seg[seg0 + pc.k], h, pc, smem + ((j + kStages - 1) % kStages) * C::STAGE, tid);
            cursor_next(p, seg0, nseg, r0, r1, pc);
        }
        cp_async_commit();

        const uint8_t *st = smem + (j % kStages) * C::STAGE;
        const int tb = cc.T * kTile;
        const int la = cc.la, le = cc.le;
        const int pos_base = p.seg[seg0 + cc.k].pos0 + tb;
        cursor_next(p, seg0, nseg, r0, r1, cc);
        if (tb + u0w >= le || tb + u0w + 16 <= la) continue;   // no valid token for this warp
        // every token of this warp's 16 valid and visible to every live row?
        const bool full = tb + u0w >= la && tb + u0w + 16 <= le && pos_base + u0w + 15 <= lim_min;

        auto chunk = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            // ---- S = Q K^T per 32-block (exact integers in fp32), scaled scores ----
            float s[2][NT][2];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int u = u0w + 8 * sub + g;              // K column this lane supplies
                float sc[MTQ][kNB][4];
#pragma unroll
                for (int bb = 0; bb < kNB; ++bb) {
                    const uint2 kb = *reinterpret_cast<const uint2 *>(st + C::K_OFF + u * kD +
                                                                      (((2 * bb + (c >> 1)) ^ g) << 4) + ((c & 1) << 3));
                    uint32_t b00, b01, b10, b11;
                    k_word_biased(kb.x, b00, b01);
                    k_word_biased(kb.y, b10, b11);
#pragma unroll
                    for (int mq = 0; mq < MTQ; ++mq) {
                        sc[mq][bb][0] = sc[mq][bb][1] = cinit[mq][bb][0];
                        sc[mq][bb][2] = sc[mq][bb][3] = cinit[mq][bb][1];
                        mma_f16_16816(sc[mq][bb], qa[mq][bb][0], b00, b01);
                        mma_f16_16816(sc[mq][bb], qa[mq][bb][1], b10, b11);
                    }
                }
                // K scales of this lane's two score columns (tokens u0w + 8sub + 2c + e)
                const int ut = u0w + 8 * sub + 2 * c;
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
                                const size_t o = ((((size_t)b * p.t_q + i) * p.n_q_heads + hq) * p.max_len + pos) * kNB;
                                int4 v;
                                v.x = (int)sc[mq][0][idx]; v.y = (int)sc[mq][1][idx];
                                v.z = (int)sc[mq][2][idx]; v.w = (int)sc[mq][3][idx];
                                *reinterpret_cast<int4 *>(p.dbg_scores + o) = v;
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
            float dv[2][2][kNB];   // [sub][e][block] V scales of this lane's B columns, 0 if invalid
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
                const int ut = u0w + 8 * sub + 2 * c;
                const uint4 vsr = *reinterpret_cast<const uint4 *>(st + C::VS_OFF + ut * kNB * 2);
                const float2 a0 = __half22float2(*reinterpret_cast<const __half2 *>(&vsr.x));
                const float2 a1 = __half22float2(*reinterpret_cast<const __half2 *>(&vsr.y));
                const float2 a2 = __half22float2(*reinterpret_cast<const __half2 *>(&vsr.z));
                const float2 a3 = __half22float2(*reinterpret_cast<const __half2 *>(&vsr.w));
                bool ok0 = true, ok1 = true;
                if (!FULL) {
                    ok0 = tb + ut >= la && tb + ut < le;
                    ok1 = tb + ut + 1 >= la && tb + ut + 1 < le;
                }
                dv[sub][0][0] = ok0 ? a0.x : 0.f; dv[sub][0][1] = ok0 ? a0.y : 0.f;
                dv[sub][0][2] = ok0 ? a1.x : 0.f; dv[sub][0][3] = ok0 ? a1.y : 0.f;
                dv[sub][1][0] = ok1 ? a2.x : 0.f; dv[sub][1][1] = ok1 ? a2.y : 0.f;
                dv[sub][1][2] = ok1 ? a3.x : 0.f; dv[sub][1][3] = ok1 ? a3.y : 0.f;
            }
#pragma unroll
            for (int bb = 0; bb < kNB; ++bb) {
                uint32_t bhi[NT][2], blo[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        const float x0 = s[sub][nt][0] * dv[sub][0][bb];
                        const float x1 = s[sub][nt][1] * dv[sub][1][bb];
                        const uint32_t hv = pack_half2(x0, x1);
                        const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hv));
                        bhi[nt][sub] = hv;
                        blo[nt][sub] = pack_half2(x0 - hf.x, x1 - hf.y);
                    }
                uint32_t t[2][4];
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    uint32_t P[4];
                    v_codes_to_half2<VT>(st + C::V_OFF, u0w + 8 * sub + g, bb, c, P);
#pragma unroll
                    for (int i = 0; i < 4; ++i) t[sub][i] = movmatrix_t(P[i]);
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint32_t a[4] = {t[0][2 * h2], t[0][2 * h2 + 1], t[1][2 * h2], t[1][2 * h2 + 1]};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16_16816(acc[2 * bb + h2][nt], a, bhi[nt][0], bhi[nt][1]);
                        mma_f16_16816(acc[2 * bb + h2][nt], a, blo[nt][0], blo[nt][1]);
                    }
                }
            }
        };
        if (full)
            chunk(std::integral_constant<bool, true>());
        else
            chunk(std::integral_constant<bool, false>());
    }

    cp_async_wait<0>();
    if constexpr (!DUMP) {

    // ---- merge the four warps' (m, l, acc) and write ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        l[nt] += __shfl_xor_sync(0xffffffffu, l[nt], 1);
        l[nt] += __shfl_xor_sync(0xffffffffu, l[nt], 2);
    }
    __syncthreads();   // every warp is done with the stage ring
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
    // Fixed merge order (warp 0 stores, warps 1..3 add in turn) so results do
    // not depend on scheduling; each (row, dim) belongs to one lane per warp.
    for (int w = 0; w < kWarps; ++w) {
        if (warp == w) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = 8 * nt + 2 * c + e;
                    if (row >= R) continue;
                    float M = -INFINITY;
#pragma unroll
                    for (int v = 0; v < kWarps; ++v) M = fmaxf(M, sm_m[v * 8 * NT + row]);
                    const float mw = sm_m[w * 8 * NT + row];
                    const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        float *o0 = &sm_o[row * kD + pv_dim<VT>(mt, g)];
                        float *o1 = &sm_o[row * kD + pv_dim<VT>(mt, g + 8)];
                        *o0 = (w == 0 ? 0.f : *o0) + acc[mt][nt][e] * f;
                        *o1 = (w == 0 ? 0.f : *o1) + acc[mt][nt][2 + e] * f;
                    }
                }
        }
        __syncthreads();
    }
    for (int row = 0; row < R; ++row) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * 8 * NT + row]);
        float Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = sm_m[w * 8 * NT + row];
            if (mw != -INFINITY) Lsum += sm_l[w * 8 * NT + row] * exp2f(mw - M);
        }
        const int i = row / gsz, hq = p.grp_q[gb + row % gsz];
        const size_t orow = ((size_t)b * p.t_q + i) * p.n_q_heads + hq;
        const bool any = Lsum > 0.f;
        const float o = any ? sm_o[row * kD + tid] / Lsum : 0.f;
        const float ls = any ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        if (p.n_split == 1) {
            p.out[orow * kD + tid] = o;
            if (tid == 0) p.lse[orow] = ls;
        } else {
            p.ws_o[(orow * p.n_split + split) * kD + tid] = o;
            if (tid == 0) p.ws_lse[orow * p.n_split + split] = ls;
        }
    }
    }
}

template <int NT, int VT>
cudaError_t launch_split_t(const AttnParams &p, bool dump, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_split, p.n_kv_heads, p.n_seqs);
    cfg.blockDim = dim3(kThreads);
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
    if (ctas_per_sm) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, kThreads, smem);
    return cudaSuccess;
}

#define KVQ_DEFINE_SPLIT_ENTRY(SUFFIX, VT)                                                   \
    cudaError_t launch_split_##SUFFIX(const AttnParams &p, int nt, bool dump, cudaStream_t s, bool pdl) \
    {                                                                                        \
        switch (nt) {                                                                        \
        case 1: return launch_split_t<1, VT>(p, dump, s, pdl);                               \
        case 2: return launch_split_t<2, VT>(p, dump, s, pdl);                               \
        case 4: return launch_split_t<4, VT>(p, dump, s, pdl);                               \
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
