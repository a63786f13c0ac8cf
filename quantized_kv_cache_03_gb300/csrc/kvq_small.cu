// kvq_small.cu -- the append/quantize kernel and the split-combine kernel.
#include "kvq_internal.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// Append-quantize.  One warp per (token, kv head) row of 128 fp16 values
// (quant_token / store_token): codes go to their place in the position's
// 16-position tile (k_tile_off / v4_tile_off / v8_tile_off): a K lane's four
// codes stay one word; q4_0 lanes 0..3 of each block pull the codes of
// elements 16.. from lanes 4..7, form bytes j = q[j] | q[j+16] << 4 and store
// them as two byte pairs; q8_0 codes are stored byte by byte (the tile
// interleaves neighbouring positions).  F16 K (KT = KVQ_K_F16): the lane's four
// fp16 K values go to their places in the 4096-byte tile as two 32-bit pairs.
// Segments of KVQ_LAYOUT_ROWS get the token's rows in element order instead
// (store_token_rows: one 32-bit word per lane and array).
// ---------------------------------------------------------------------------
template <int VT, int KT>
__global__ void __launch_bounds__(128) append_kernel(const __grid_constant__ AppendParams p)
{
    pdl_wait();      // inputs come from earlier kernels; the cache may still be read by one
    pdl_trigger();
    const AppendEntry &e = p.e[blockIdx.y];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = p.n_kv_heads;
    const int row = blockIdx.x * 4 + warp;
    const int tok = row / H, h = row - tok * H;
    if (tok >= e.n) return;   // warp-uniform
    const size_t src = ((size_t)(e.src + tok) * H + h) * kD;
    const int u = (e.dst + tok) % kWTile;                      // position in its tile
    const size_t tile = (size_t)h * e.cap + e.dst + tok - u;    // first row of the tile
    const TokenRow t = quant_token<VT, KT>(p.k16 + src, p.v16 + src, lane);
    constexpr int VCODE = VT == KVQ_V_Q4_0 ? kD / 2 : kD;
    if (KT == KVQ_K_I8 && e.layout == KVQ_LAYOUT_ROWS)   // the token's own rows, element order
        store_token_rows<VT>(t, lane, e.kq + (tile + u) * kD, e.ks + (tile + u) * kNB, e.vq + (tile + u) * VCODE,
                             e.vs + (tile + u) * kNB);
    else
        store_token<VT, KT>(t, u, lane, e.kq + tile * kD * (KT == KVQ_K_F16 ? 2 : 1), e.ks + (tile + u) * kNB,
                            e.vq + tile * VCODE, e.vs + (tile + u) * kNB);
}

cudaError_t launch_append(const AppendParams &p, int v_type, int k_type, int max_rows, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((max_rows + 3) / 4, p.n_entries);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (k_type == KVQ_K_F16)
        return (v_type == KVQ_V_Q4_0) ? cudaLaunchKernelEx(&cfg, append_kernel<KVQ_V_Q4_0, KVQ_K_F16>, p)
                                      : cudaLaunchKernelEx(&cfg, append_kernel<KVQ_V_Q8_0, KVQ_K_F16>, p);
    return (v_type == KVQ_V_Q4_0) ? cudaLaunchKernelEx(&cfg, append_kernel<KVQ_V_Q4_0, KVQ_K_I8>, p)
                                  : cudaLaunchKernelEx(&cfg, append_kernel<KVQ_V_Q8_0, KVQ_K_I8>, p);
}

// ---------------------------------------------------------------------------
// Split combine: per query row, M = max_s lse_s, w_s = exp(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s, lse = M + log(sum_s w_s).  One CTA per row
// (rows of every group of the launch in one grid).  Warp w takes splits
// w, w + 8, ... four at a time, loading their lse and o (each lane four head
// dims, float4) in one round trip, and keeps a running (max, weight sum,
// weighted o) with rescaling; warp 0 then merges the eight warp states in a
// fixed order.  Splits with lse = -inf (no visible position) weigh 0 and their
// o is never used.
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const __grid_constant__ CombineParams p)
{
    __shared__ float sm_m[kCombineWarps], sm_w[kCombineWarps];
    __shared__ float4 part[kCombineWarps][32];
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if ((int)blockIdx.x >= p.grp[k].row0) gi = k;
    const CombineGroup &G = p.grp[gi];
    const int row = (int)blockIdx.x - G.row0, warp = threadIdx.x >> 5, lane = threadIdx.x & 31, n = G.n_split;
    pdl_wait();
    pdl_trigger();
    const float *ls = G.ws_lse + (size_t)row * n;
    const float4 *o = reinterpret_cast<const float4 *>(G.ws_o + (size_t)row * n * kD) + lane;
    float m = -INFINITY, W = 0.f;
    bool poisoned = false;   // a split wrote NaN (its CTA lost a copy stage)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = warp; s0 < n; s0 += 4 * kCombineWarps) {
        float lv[4];
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int s = s0 + k * kCombineWarps;
            lv[k] = (s < n) ? ls[s] : -INFINITY;
            v[k] = (s < n) ? o[(size_t)s * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
            poisoned |= lv[k] != lv[k];
        }
        const float mx = fmaxf(fmaxf(m, fmaxf(lv[0], lv[1])), fmaxf(lv[2], lv[3]));
        if (mx == -INFINITY) continue;
        const float a = (m == -INFINITY) ? 0.f : expf(m - mx);
        W *= a;
        acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float w = (lv[k] == -INFINITY) ? 0.f : expf(lv[k] - mx);
            W += w;
            if (w != 0.f) {
                acc.x = fmaf(w, v[k].x, acc.x);
                acc.y = fmaf(w, v[k].y, acc.y);
                acc.z = fmaf(w, v[k].z, acc.z);
                acc.w = fmaf(w, v[k].w, acc.w);
            }
        }
        m = mx;
    }
    if (poisoned) {   // m = +inf and W = NaN make the merged row NaN
        m = INFINITY;
        W = __int_as_float(0x7fc00000);
    }
    if (lane == 0) {
        sm_m[warp] = m;
        sm_w[warp] = W;
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, sm_m[w]);
        float Wt = 0.f;
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) {
            if (sm_m[w] == -INFINITY) continue;
            const float f = expf(sm_m[w] - M);
            Wt = fmaf(sm_w[w], f, Wt);
            const float4 q = part[w][lane];
            t.x = fmaf(q.x, f, t.x); t.y = fmaf(q.y, f, t.y); t.z = fmaf(q.z, f, t.z); t.w = fmaf(q.w, f, t.w);
        }
        const bool any = !(Wt <= 0.f);   // a NaN weight (a poisoned partial) keeps the row NaN
        const float inv = any ? 1.f / Wt : 0.f;
        reinterpret_cast<float4 *>(G.out + (size_t)row * kD)[lane] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
        if (lane == 0) G.lse[row] = any ? M + logf(Wt) : -INFINITY;
    }
}

// The same merge for launches whose rows have at most kNarrowSplits splits
// each (long query chunks: thousands of rows, two splits; the long-context
// step: 56 rows, 12 splits): one warp per row, eight rows per CTA, the splits
// merged one after another in split order with the same running (max, weight
// sum, weighted o).  One CTA per row would leave most warps idle and make the
// launch a stream of tiny CTAs.  Measured: the prefill chunk's 16384 rows x 2
// splits 31 -> 8 us; the long-context step 65.78 -> 65.47 us; 32 rows x 16
// splits slower this way (11.85 -> 12.5 us per step), so more splits keep
// one CTA per row.
constexpr int kNarrowSplits = 12;

// NS: the most splits a row of the launch has room for (4 or kNarrowSplits):
// every lane loads NS slots, so a launch of two-split rows takes the small form.
template <int NS>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_rows_kernel(const __grid_constant__ CombineParams p,
                                                                          int n_rows)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (int)blockIdx.x * kCombineWarps + warp;
    pdl_wait();
    pdl_trigger();
    if (r >= n_rows) return;
    int gi = 0;
#pragma unroll 1
    for (int k = 1; k < p.n_groups; ++k)
        if (r >= p.grp[k].row0) gi = k;
    const CombineGroup &G = p.grp[gi];
    const int row = r - G.row0, n = G.n_split;
    const float *ls = G.ws_lse + (size_t)row * n;
    const float4 *o = reinterpret_cast<const float4 *>(G.ws_o + (size_t)row * n * kD) + lane;
    float lv[NS];
    float4 v[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) {   // every split's lse and o in one round trip
        lv[k] = (k < n) ? ls[k] : -INFINITY;
        v[k] = (k < n) ? o[(size_t)k * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = -INFINITY, W = 0.f;
    bool poisoned = false;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NS; ++k) {
        poisoned |= lv[k] != lv[k];
        if (lv[k] == -INFINITY || lv[k] != lv[k]) continue;
        const float mx = fmaxf(m, lv[k]);
        const float a = (m == -INFINITY) ? 0.f : expf(m - mx), w = expf(lv[k] - mx);
        W = fmaf(W, a, w);
        acc.x = fmaf(w, v[k].x, acc.x * a);
        acc.y = fmaf(w, v[k].y, acc.y * a);
        acc.z = fmaf(w, v[k].z, acc.z * a);
        acc.w = fmaf(w, v[k].w, acc.w * a);
        m = mx;
    }
    if (poisoned) {   // a split that lost a copy stage: the merged row is NaN
        m = INFINITY;
        W = __int_as_float(0x7fc00000);
    }
    const bool any = !(W <= 0.f);
    const float inv = any ? 1.f / W : 0.f;
    reinterpret_cast<float4 *>(G.out + (size_t)row * kD)[lane] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (lane == 0) G.lse[row] = any ? m + logf(W) : -INFINITY;
}

cudaError_t launch_combine(const CombineParams &p, int n_rows, cudaStream_t s, bool pdl)
{
    int max_split = 0;
    for (int k = 0; k < p.n_groups; ++k) max_split = max(max_split, p.grp[k].n_split);
    const bool narrow = max_split <= kNarrowSplits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(narrow ? (n_rows + kCombineWarps - 1) / kCombineWarps : n_rows);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (narrow && max_split <= 4) return cudaLaunchKernelEx(&cfg, combine_rows_kernel<4>, p, n_rows);
    if (narrow) return cudaLaunchKernelEx(&cfg, combine_rows_kernel<kNarrowSplits>, p, n_rows);
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace kvq
