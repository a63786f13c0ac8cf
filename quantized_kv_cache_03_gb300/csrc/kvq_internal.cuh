// kvq_internal.cuh -- launch-parameter structs and sm_103a device helpers shared
// by the CUDA translation units of libkvq.so.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kD = KVQ_HEAD_DIM;        // head dim
constexpr int kNB = kD / KVQ_QBLOCK;    // 32-blocks per head row (4)
constexpr int kWTile = 16;              // positions per warp pipeline stage

#ifndef KVQ_WARPS_NT1
#define KVQ_WARPS_NT1 16   // warps per CTA of the <= 8-row kernels (128 registers: one CTA per SM)
#endif
#ifndef KVQ_WARPS_NTX
#define KVQ_WARPS_NTX 4    // warps per CTA of the 16- and 32-row kernels (more registers per thread)
#endif
// Warps per split CTA for nt 8-row query tiles; each warp streams its own
// contiguous sub-range of the split, so split chunks are rounded to a multiple
// of the CTA's warps * kWTile positions.  The 8-row kernel also comes with half
// as many warps (two CTAs per SM, the same warps per SM), for launches that
// take more than one wave of full CTAs: their work is then dealt in pieces
// half as large, which evens out the last wave.
constexpr int split_warps(int nt) { return nt == 1 ? KVQ_WARPS_NT1 : KVQ_WARPS_NTX; }
constexpr int kWarpsHalf = KVQ_WARPS_NT1 / 2;
constexpr int kPrefillRows = 128;       // query rows per CTA of the tcgen05 kernel
constexpr int kPrefillPositions = 64;   // positions per KV tile of the tcgen05 kernel
constexpr int kMaxSegsLaunch = 64;      // segment-table entries per launch
constexpr int kMaxSeqsLaunch = 64;      // sequences per launch

// ------------------------------------------------------------ tile layout --
// A segment stores each kv head's positions in tiles of kWTile = 16: tile T of
// head h holds positions 16T..16T+15 and starts (h*cap + 16T) rows into each
// array, so a tile of every array is one contiguous run of bytes (K codes 2048,
// V codes 1024 (q4_0) or 2048 (q8_0), K and V scales 128 each) that a single
// bulk copy moves.  Scales keep the plain [position][block] fp16 order.  The
// code bytes of a tile are permuted so that the 16-byte word at
// i*512 + lane*16 is the lane's i-th shared-memory load (lane = 4g + c of the
// attention kernel's mma fragments); the bytes themselves are unchanged.
// With u the position in the tile (sub = u/8, gu = u%8, cu = (u%8)/2, e = u%2)
// and j the byte of the logical row:
//   K      (j < 128, block bb = j/32):
//          ((2 sub + bb/2) * 32 + 4 gu + (j%32)/8) * 16 + 8 (bb%2) + j%8
//   V q4_0 (j < 64, bb = j/16, jj = j%16):
//          (sub * 32 + 4 (jj/2) + cu) * 16 + 4 bb + 2 e + jj%2
//   V q8_0 (j < 128, bb = j/32, jj = j%32):
//          ((2 sub + bb/2) * 32 + 4 (jj/4) + cu) * 16 + 8 (bb%2) + 4 ((jj%4)/2) + 2 (jj%2) + e
// so a K load gives one position's 8 codes of two blocks, a q4_0 load the code
// bytes 2g, 2g+1 of positions (t, t+1) of all four blocks, and a q8_0 load
// codes 4g..4g+3 of positions (t, t+1) of two blocks, (t, t+1) interleaved.
__host__ __device__ constexpr int k_tile_off(int u, int j)
{
    return ((2 * (u / 8) + j / 64) * 32 + 4 * (u % 8) + (j % 32) / 8) * 16 + 8 * ((j / 32) % 2) + j % 8;
}
__host__ __device__ constexpr int v4_tile_off(int u, int j)
{
    return ((u / 8) * 32 + 4 * ((j % 16) / 2) + (u % 8) / 2) * 16 + 4 * (j / 16) + 2 * (u % 2) + j % 2;
}
// F16 K: byte offset of fp16 element j of token u in a 4096-byte tile, the
// mma A-fragment order (16-byte word at ks*512 + lane*16 holds the four
// registers of k16 step ks for lane = 4*(u%8) + (j%8)/2: rows u, u+8 of
// elements 2c, 2c+1 and 2c+8, 2c+9).
__host__ __device__ constexpr int k16_tile_off(int u, int j)
{
    return (j / 16) * 512 + (4 * (u % 8) + (j % 8) / 2) * 16 + 4 * (u / 8 + 2 * ((j % 16) / 8)) + 2 * (j % 2);
}
__host__ __device__ constexpr int v8_tile_off(int u, int j)
{
    return ((2 * (u / 8) + j / 64) * 32 + 4 * ((j % 32) / 4) + (u % 8) / 2) * 16 + 8 * ((j / 32) % 2) +
           4 * ((j % 4) / 2) + 2 * (j % 2) + u % 2;
}

// One segment as the attention kernel sees it (device pointers of kv head 0;
// head h starts h*cap tokens further).
struct SegDesc {
    const uint8_t *kq;    // [Hkv][cap/16] tiles of 2048 code bytes
    const uint16_t *ks;   // [Hkv][cap][kNB] fp16 bits
    const uint8_t *vq;    // [Hkv][cap/16] tiles of 1024 (q4_0) or 2048 (q8_0) code bytes
    const uint16_t *vs;   // [Hkv][cap][kNB]
    int pos0;             // absolute position of token 0
    int cap;              // tokens, multiple of KVQ_SEG_ALIGN
    int layout;           // kvq_layout of the code bytes
};

// One work group of a split launch: sequences [b0, b0 + n_seqs) of one cache
// of one decode call.  A launch runs up to kMaxGroups groups (of one or more
// caches) in a single 1-D grid; CTA cta0 + ((b * n_kv_heads + h) * n_split + s)
// * n_rt + rt of the group attends split s of kv head h of its sequence b for
// row tile rt (the fastest-varying index, so a kv head's row tiles stream the
// same positions side by side).
struct GroupDesc {
    const uint16_t *q;                     // [n_seqs][t_q][Hq][kD] fp16 bits
    const int *seq_lens;                   // [n_seqs]
    float *out;                            // [n_seqs][t_q][Hq][kD]       (n_split == 1)
    float *lse;                            // [n_seqs][t_q][Hq]
    float *ws_o;                           // [n_seqs][t_q][Hq][n_split][kD] (n_split > 1)
    float *ws_lse;                         // [n_seqs][t_q][Hq][n_split]
    int8_t *dbg_qc;                        // test hook outputs (DUMP kernels only)
    uint16_t *dbg_qs;
    int32_t *dbg_scores;
    const uint16_t *k_new, *v_new;         // [n_seqs][t_q][Hkv][kD] fp16 tokens appended by this call, or null
    int cta0;                              // first CTA of the group
    int seq0;                              // first entry of seq_seg0 / seq_nseg
    int head0;                             // first entry of grp_begin (this cache's kv heads)
    int n_seqs, n_kv_heads, n_q_heads, t_q, causal;
    int max_len;                           // positions >= max_len are ignored
    int n_split, chunk;                    // split s covers [s*chunk, (s+1)*chunk) ...
    int chunk0;                            // ... when chunk0 == chunk; else split 0 covers [0, chunk0)
                                           // and split s >= 1 [chunk0 + (s-1)*chunk, chunk0 + s*chunk)
                                           // (the tcgen05 kernel's uneven split; the split kernel
                                           // always gets chunk0 == chunk)
    int split_major;                       // CTA order split, seq, kv head, row tile (else seq, kv head,
                                           // split, row tile); tcgen05 kernel only
    int n_rt;                              // row tiles of 8*NT query rows per kv head
    float qk_scale_log2;                   // sm_scale * log2(e)
};

constexpr int kMaxGroups = 8;              // work groups per launch
constexpr int kMaxHeadTab = 512;           // query-head list entries per launch

struct AttnParams {
    SegDesc seg[kMaxSegsLaunch];
    uint8_t seq_seg0[kMaxSeqsLaunch];      // first table entry of each sequence
    uint8_t seq_nseg[kMaxSeqsLaunch];
    int app_pos[kMaxSeqsLaunch];           // absolute position of a sequence's first appended token
    uint16_t grp_q[kMaxHeadTab];           // query heads listed kv head by kv head
    uint16_t grp_begin[kMaxHeadTab + kMaxGroups];   // kv head h of group g owns
                                           // grp_q[grp_begin[head0 + h] .. grp_begin[head0 + h + 1])
    GroupDesc grp[kMaxGroups];
    int n_groups;
    unsigned int *timeouts;                // bumped when a copy wait gives up (never in a correct run)
};

// Split combine of one group: rows [row0, row0 + n_rows) of the launch.
struct CombineGroup {
    const float *ws_o;
    const float *ws_lse;
    float *out;
    float *lse;
    int row0;                              // first CTA (row) of the group
    int n_split;
};

struct CombineParams {
    CombineGroup grp[kMaxGroups];
    int n_groups;
};

struct AppendEntry {
    uint8_t *kq;
    uint16_t *ks;
    uint8_t *vq;
    uint16_t *vs;
    int cap;                               // tokens
    int dst;                               // first token slot written
    int src;                               // first input token row
    int n;                                 // tokens
    int layout;                            // kvq_layout of the segment
};

struct AppendParams {
    AppendEntry e[kMaxSeqsLaunch];
    const uint16_t *k16;                   // [sum n][Hkv][kD]
    const uint16_t *v16;
    int n_entries;
    int n_kv_heads;
};

// ------------------------------------------------------------ host launchers --
// Implemented in kvq_small.cu / kvq_attn_q4.cu / kvq_attn_q8.cu / kvq_prefill_q*.cu.
// n_tiles8 = query rows per kv head rounded up to 1, 2 or 4 tiles of 8; warps =
// split_warps(n_tiles8), or kWarpsHalf with one tile.  k_type selects the K
// format (kvq_ktype); dump kernels exist for KVQ_K_I8 at split_warps only.
cudaError_t launch_append(const AppendParams &p, int v_type, int k_type, int max_rows, cudaStream_t s, bool pdl);
cudaError_t launch_combine(const CombineParams &p, int n_rows, cudaStream_t s, bool pdl);
// Split-kernel flavours: the decode kernel; the score-dump test hook (int8 K,
// split_warps(n_tiles8) warps); the lose-stage test hook (int8 K, one 8-row
// tile, 16 warps), in which one stage's wait runs out on purpose.
constexpr int kModeDecode = 0, kModeDump = 1, kModeLoseStage = 2;
cudaError_t launch_split_q4(const AttnParams &p, int n_tiles8, int warps, int k_type, int n_ctas, int mode,
                            cudaStream_t s, bool pdl);
cudaError_t launch_split_q8(const AttnParams &p, int n_tiles8, int warps, int k_type, int n_ctas, int mode,
                            cudaStream_t s, bool pdl);
cudaError_t prepare_split_q4(int n_tiles8, int warps, int k_type, int mode, int *ctas_per_sm);
cudaError_t prepare_split_q8(int n_tiles8, int warps, int k_type, int mode, int *ctas_per_sm);
// tcgen05 kernel for long query chunks (kvq_prefill_q4.cu / kvq_prefill_q8.cu):
// 128 query rows per CTA, one CTA per SM; dump selects its test-hook flavour
// (query codes and raw block scores instead of out / lse).
cudaError_t launch_prefill_q4(const AttnParams &p, int n_ctas, bool dump, cudaStream_t s, bool pdl);
cudaError_t launch_prefill_q8(const AttnParams &p, int n_ctas, bool dump, cudaStream_t s, bool pdl);
cudaError_t prepare_prefill_q4();
cudaError_t prepare_prefill_q8();

// ------------------------------------------------------------- device helpers --

// Programmatic dependent launch: wait for the producing grid (and its memory)
// before the first read of anything an earlier kernel wrote.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next PDL-launched grid in the stream to be scheduled.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier + bulk async copy (one elected lane issues, the warp waits) ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Make barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n fence.proxy.async.shared::cta;" ::: "memory");
}
// Order this thread's earlier generic-proxy shared accesses before later
// async-proxy ones (a bulk copy into a stage the warp has just read).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Issued by a converged warp: every lane passes the same (warp-uniform)
// operands and one lane, elected inside the asm, issues.  (Issuing from inside
// a lane-0 branch costs more per instruction: the uniform operands have to be
// taken out of a divergent lane.)
// One arrival that also announces tx bytes still to land on the barrier.
__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint32_t bar, uint32_t tx)
{
    asm volatile("{\n .reg .pred e;\n .reg .b64 st;\n elect.sync _|e, 0xffffffff;\n"
                 " @e mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar), "r"(tx)
                 : "memory");
}
// Contiguous global -> shared copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) that completes its bytes on barrier `bar`.
__device__ __forceinline__ void bulk_g2s_w(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
                 " @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n}"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// Wait for phase `parity` of the barrier to complete, giving up after
// kMbarSpins polls (each poll may suspend the thread for a short while).
constexpr uint32_t kMbarSpins = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t spins = kMbarSpins)
{
    for (uint32_t i = 0; i < spins; ++i) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done) return true;
    }
    return false;
}



// The pieces of a sequence's segments that fall in [r0, r1), walked in order
// in tiles of kWTile positions: T is the next tile of segment k, Tend the end of
// the piece, and gk..gvs point at tile T's data in the four arrays.
struct Walk {
    int k;            // segment table entry (relative to the sequence's first); nseg when done
    int T, Tend;      // next tile inside the segment, end tile (exclusive) of the piece
    int la, le;       // local range [la, le) of the current piece
    int pos0;
    int rows;         // the segment keeps KVQ_LAYOUT_ROWS (rows in element order)
    const uint8_t *gk, *gks, *gv, *gvs;
};

__device__ __forceinline__ void walk_seek(const AttnParams &p, int seg0, int nseg, int h, int r0, int r1, int k,
                                          int vcode, Walk &w, int kcode = kD)
{
    for (w.k = k; w.k < nseg; ++w.k) {
        const SegDesc &s = p.seg[seg0 + w.k];
        const int end = (w.k + 1 < nseg) ? p.seg[seg0 + w.k + 1].pos0 : s.pos0 + s.cap;
        const int a = max(r0, s.pos0), e = min(min(r1, end), s.pos0 + s.cap);
        if (a < e) {
            w.la = a - s.pos0;
            w.le = e - s.pos0;
            w.T = w.la / kWTile;
            w.Tend = (w.le + kWTile - 1) / kWTile;
            w.pos0 = s.pos0;
            w.rows = s.layout == KVQ_LAYOUT_ROWS;
            const size_t row = (size_t)h * s.cap + (size_t)w.T * kWTile;
            w.gk = reinterpret_cast<const uint8_t *>(s.kq) + row * kcode;
            w.gks = reinterpret_cast<const uint8_t *>(s.ks) + row * kNB * 2;
            w.gv = s.vq + row * vcode;
            w.gvs = reinterpret_cast<const uint8_t *>(s.vs) + row * kNB * 2;
            return;
        }
    }
}


// D = A(16x16 f16, row) * B(16x8 f16, col) + C, C given as four floats (bit patterns).
__device__ __forceinline__ void mma_f16_16816_c4(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                                 const uint4 &c)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(__uint_as_float(c.x)),
          "f"(__uint_as_float(c.y)), "f"(__uint_as_float(c.z)), "f"(__uint_as_float(c.w)));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic): one instruction for two lanes
// of independent fp32 work, rounding as the scalar operation.
__device__ __forceinline__ unsigned long long f2_bits(float2 a) { return *reinterpret_cast<unsigned long long *>(&a); }
__device__ __forceinline__ float2 f2_from(unsigned long long a) { return *reinterpret_cast<float2 *>(&a); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_from(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_from(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return f2_from(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return f2_from(r);
}

// Transpose an 8x8 matrix of 16-bit elements held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// 2^x (hardware approximation, flushes subnormals).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// int8 rule of one element given its block scale s (fp32 copy of the fp16 scale).
__device__ __forceinline__ int quant_i8(float x, float s)
{
    if (s == 0.f) return 0;
    float c = roundf(__fdiv_rn(x, s));          // correctly rounded quotient, ties away
    return (int)fminf(fmaxf(c, -127.f), 127.f);
}

// q4_0 rule of one element given d (fp32 copy of the fp16 scale).
__device__ __forceinline__ int quant_q4(float x, float d)
{
    if (d == 0.f) return 8;
    float c = roundf(__fdiv_rn(x, d)) + 8.f;
    return (int)fminf(fmaxf(c, 0.f), 15.f);
}


// ---- one (token, kv head) row through the append rules (warp-wide) ----
// Lane l holds elements 4l..4l+3, so lanes 8b..8b+7 hold 32-block b and a
// 3-step xor shuffle gives the block absmax.
__device__ __forceinline__ float block_absmax(const float (&x)[4])
{
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    return a;
}

__device__ __forceinline__ void load4h(const uint16_t *p, float (&x)[4])
{
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// int8 rule on one row: returns this lane's packed word and the block scale bits.
__device__ __forceinline__ uint32_t quant_row_i8(const float (&x)[4], uint16_t &s16)
{
    const float a = block_absmax(x);
    const __half sh = __float2half_rn(__fdiv_rn(a, 127.f));
    const float s = __half2float(sh);
    s16 = __half_as_ushort(sh);
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) w |= (uint32_t)(quant_i8(x[k], s) & 0xff) << (8 * k);
    return w;
}

// A quantized (token, kv head) row as the lanes hold it: kw = K codes 4l..4l+3;
// ks = block (l/8) K scale bits; vw = q8_0 codes 4l..4l+3, or for q4_0 lanes
// with l%8 < 4 the code bytes 4(l%4)..+3 of block l/8 (byte j = q[j] | q[j+16] << 4);
// vs = block (l/8) V scale bits.
struct TokenRow {
    uint32_t kw, vw;
    uint16_t ks, vs;
    uint32_t kw2;   // F16 K: kw, kw2 = the lane's four fp16 K values
};

template <int VT, int KT = KVQ_K_I8>
__device__ __forceinline__ TokenRow quant_token(const uint16_t *k_row, const uint16_t *v_row, int lane)
{
    TokenRow t;
    float x[4];
    if (KT == KVQ_K_F16) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(k_row + lane * 4);
        t.kw = raw.x;
        t.kw2 = raw.y;
        t.ks = 0;
    } else {
        load4h(k_row + lane * 4, x);
        t.kw = quant_row_i8(x, t.ks);
        t.kw2 = 0;
    }
    load4h(v_row + lane * 4, x);
    if (VT == KVQ_V_Q8_0) {
        t.vw = quant_row_i8(x, t.vs);
    } else {
        const float a = block_absmax(x);
        const __half dh = __float2half_rn(a * 0.125f);   // absmax/8, exact before rounding
        const float d = __half2float(dh);
        uint32_t q = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) q |= (uint32_t)quant_q4(x[k], d) << (8 * k);
        const uint32_t qhi = __shfl_down_sync(0xffffffffu, q, 4);   // elements 16.. of the block
        t.vw = q | (qhi << 4);
        t.vs = __half_as_ushort(dh);
    }
    return t;
}

// Store a quantized row at tile position u of the code tiles kt / vt (K codes,
// V codes) and at scale rows ksr / vsr (4 fp16 each), in the cache's tile order.
// Works for a tile in global memory and for a staged copy in shared memory.
template <int VT, int KT = KVQ_K_I8>
__device__ __forceinline__ void store_token(const TokenRow &t, int u, int lane, uint8_t *kt, uint16_t *ksr,
                                            uint8_t *vt, uint16_t *vsr)
{
    if (KT == KVQ_K_F16) {   // elements 4l, 4l+1 and 4l+2, 4l+3: one 32-bit pair each
        *reinterpret_cast<uint32_t *>(kt + k16_tile_off(u, 4 * lane)) = t.kw;
        *reinterpret_cast<uint32_t *>(kt + k16_tile_off(u, 4 * lane + 2)) = t.kw2;
    } else {
        *reinterpret_cast<uint32_t *>(kt + k_tile_off(u, 4 * lane)) = t.kw;
        if ((lane & 7) == 0) ksr[lane >> 3] = t.ks;
    }
    if (VT == KVQ_V_Q8_0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) vt[v8_tile_off(u, 4 * lane + k)] = (uint8_t)(t.vw >> (8 * k));
    } else if ((lane & 7) < 4) {
        const int j = 16 * (lane >> 3) + 4 * (lane & 3);
        *reinterpret_cast<uint16_t *>(vt + v4_tile_off(u, j)) = (uint16_t)t.vw;
        *reinterpret_cast<uint16_t *>(vt + v4_tile_off(u, j + 2)) = (uint16_t)(t.vw >> 16);
    }
    if ((lane & 7) == 0) vsr[lane >> 3] = t.vs;
}

// The same row stored in KVQ_LAYOUT_ROWS order (global memory): kr, vr point
// at the token's K and V code rows, ksr / vsr at its scale rows.
template <int VT>
__device__ __forceinline__ void store_token_rows(const TokenRow &t, int lane, uint8_t *kr, uint16_t *ksr, uint8_t *vr,
                                                 uint16_t *vsr)
{
    *reinterpret_cast<uint32_t *>(kr + 4 * lane) = t.kw;
    if ((lane & 7) == 0) ksr[lane >> 3] = t.ks;
    if (VT == KVQ_V_Q8_0) {
        *reinterpret_cast<uint32_t *>(vr + 4 * lane) = t.vw;
    } else if ((lane & 7) < 4) {   // bytes 4(l%4)..+3 of block l/8
        *reinterpret_cast<uint32_t *>(vr + 16 * (lane >> 3) + 4 * (lane & 3)) = t.vw;
    }
    if ((lane & 7) == 0) vsr[lane >> 3] = t.vs;
}

// ---- a staged tile of a KVQ_LAYOUT_ROWS segment -> the tile order ----
// One warp permutes a tile's code bytes in shared memory in place: every lane
// loads its 16-byte pieces of the row-order tile, the warp synchronizes, and
// the lanes store them at their tile-order offsets (8-byte runs for K, 2-byte
// runs for q4_0; for q8_0 the bytes of tokens 2i and 2i + 1 interleave, so a
// lane pairs the same 4 bytes of both rows into one 8-byte run).
static __device__ __noinline__ void rows_to_tile_k(uint8_t *t, int lane)
{
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = *reinterpret_cast<const uint4 *>(t + (lane + 32 * k) * 16);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int q = lane + 32 * k, u = q >> 3, j = (q & 7) * 16;   // token u, bytes j..j+15 of its row
        *reinterpret_cast<uint2 *>(t + k_tile_off(u, j)) = make_uint2(v[k].x, v[k].y);
        *reinterpret_cast<uint2 *>(t + k_tile_off(u, j + 8)) = make_uint2(v[k].z, v[k].w);
    }
    __syncwarp();
}

template <int VT>
__device__ __noinline__ void rows_to_tile_v(uint8_t *t, int lane)
{
    if (VT == KVQ_V_Q4_0) {
        uint4 v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) v[k] = *reinterpret_cast<const uint4 *>(t + (lane + 32 * k) * 16);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int q = lane + 32 * k, u = q >> 2, bb = q & 3;   // token u, block bb (16 bytes)
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int e = 0; e < 8; ++e)   // bytes 2e, 2e + 1 of the block
                *reinterpret_cast<uint16_t *>(t + v4_tile_off(u, 16 * bb + 2 * e)) = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
        }
    } else {
        uint4 a[2], b[2];   // the same 16 bytes of tokens 2p and 2p + 1
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int q = lane + 32 * k, p = q >> 3, c16 = q & 7;
            a[k] = *reinterpret_cast<const uint4 *>(t + (2 * p) * kD + 16 * c16);
            b[k] = *reinterpret_cast<const uint4 *>(t + (2 * p + 1) * kD + 16 * c16);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int q = lane + 32 * k, p = q >> 3, c16 = q & 7;
            const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
#pragma unroll
            for (int w = 0; w < 4; ++w)   // bytes j..j+3 of both rows, interleaved token by token
                *reinterpret_cast<uint2 *>(t + v8_tile_off(2 * p, 16 * c16 + 4 * w)) =
                    make_uint2(__byte_perm(wa[w], wb[w], 0x5140), __byte_perm(wa[w], wb[w], 0x7362));
        }
    }
    __syncwarp();
}

}  // namespace kvq
