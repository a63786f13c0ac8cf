// kvq_api.cu -- the C ABI of libkvq.so: argument validation, segment-table
// marshalling, split policy and kernel launches.  No allocation, and no host
// sync except in kvq_wait_timeouts.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvq_internal.cuh"

using namespace kvq;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int n_sms = 0;
    int ctas[2][5] = {};   // [v_type][n_tiles8] resident split CTAs per SM
    unsigned int *timeouts = nullptr;   // device address of g_wait_timeouts
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
}  // namespace

// Waits in the attention kernel that gave up (see kvq_wait_timeouts).
static __device__ unsigned int g_wait_timeouts;

namespace {

// Device attributes and kernel attributes, once per device.
kvq_status device_setup(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KVQ_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_UNSUPPORTED;
        }
        if (major != 10 || minor != 3) return KVQ_ERR_UNSUPPORTED;   // built for sm_103a only
        const int nts[3] = {1, 2, 4};
        for (int i = 0; i < 3; ++i) {
            const int nt = nts[i];
            if (prepare_split_q4(nt, false, &d.ctas[KVQ_V_Q4_0][nt]) != cudaSuccess ||
                prepare_split_q8(nt, false, &d.ctas[KVQ_V_Q8_0][nt]) != cudaSuccess ||
                prepare_split_q4(nt, true, nullptr) != cudaSuccess ||
                prepare_split_q8(nt, true, nullptr) != cudaSuccess) {
                cudaGetLastError();
                return KVQ_ERR_CUDA;
            }
        }
        void *t = nullptr;
        if (cudaGetSymbolAddress(&t, g_wait_timeouts) != cudaSuccess || !t) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
        d.timeouts = static_cast<unsigned int *>(t);
        d.ready = true;
    }
    *out = &d;
    return KVQ_OK;
}

bool pdl_enabled()
{
    const char *e = std::getenv("KVQ_PDL");
    return !(e && e[0] == '0');
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

const kvq_segment &seg_of(const kvq_cache *c, int b, int k) { return c->segs[(size_t)b * c->max_segs + k]; }

// Shape and segment-table checks shared by every entry point.
kvq_status check_cache(const kvq_cache *c)
{
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (c->n_seqs < 0 || c->n_kv_heads < 1 || c->n_kv_heads > KVQ_MAX_HEADS || c->max_segs < 1)
        return KVQ_ERR_INVALID_ARG;
    if (c->v_type != KVQ_V_Q4_0 && c->v_type != KVQ_V_Q8_0) return KVQ_ERR_INVALID_ARG;
    if (c->head_dim != KVQ_HEAD_DIM) return c->head_dim % KVQ_QBLOCK ? KVQ_ERR_INVALID_ARG : KVQ_ERR_UNSUPPORTED;
    if (c->n_seqs == 0) return KVQ_OK;
    if (!c->n_segs || !c->segs) return KVQ_ERR_INVALID_ARG;
    for (int b = 0; b < c->n_seqs; ++b) {
        const int ns = c->n_segs[b];
        if (ns < 0 || ns > c->max_segs || ns > kMaxSegsLaunch) return KVQ_ERR_INVALID_ARG;
        for (int k = 0; k < ns; ++k) {
            const kvq_segment &s = seg_of(c, b, k);
            if (!s.k_q || !s.k_s || !s.v_q || !s.v_s) return KVQ_ERR_INVALID_ARG;
            if (!aligned16(s.k_q) || !aligned16(s.k_s) || !aligned16(s.v_q) || !aligned16(s.v_s))
                return KVQ_ERR_INVALID_ARG;
            if (s.cap <= 0 || s.cap % KVQ_SEG_ALIGN || s.len < 0 || s.len > s.cap) return KVQ_ERR_INVALID_ARG;
            const long long expect = k == 0 ? 0 : (long long)seg_of(c, b, k - 1).pos0 + seg_of(c, b, k - 1).len;
            if (s.pos0 != expect) return KVQ_ERR_INVALID_ARG;
            if ((long long)s.pos0 + s.cap > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;
        }
    }
    return KVQ_OK;
}

// Query-head groups per kv head from head_map (host) or contiguous groups.
kvq_status build_groups(const kvq_cache *c, int n_q_heads, const int32_t *head_map, int t_q, AttnParams &p,
                        int &max_rows)
{
    const int H = c->n_kv_heads;
    if (n_q_heads < 1 || n_q_heads > KVQ_MAX_HEADS) return KVQ_ERR_INVALID_ARG;
    std::vector<int> kv(n_q_heads);
    if (head_map) {
        for (int h = 0; h < n_q_heads; ++h) {
            if (head_map[h] < 0 || head_map[h] >= H) return KVQ_ERR_INVALID_ARG;
            kv[h] = head_map[h];
        }
    } else {
        if (n_q_heads % H) return KVQ_ERR_INVALID_ARG;
        const int gsz = n_q_heads / H;
        for (int h = 0; h < n_q_heads; ++h) kv[h] = h / gsz;
    }
    int n = 0, gmax = 0;
    for (int k = 0; k < H; ++k) {
        p.grp_begin[k] = (uint16_t)n;
        for (int h = 0; h < n_q_heads; ++h)
            if (kv[h] == k) p.grp_q[n++] = (uint8_t)h;
        gmax = std::max(gmax, n - (int)p.grp_begin[k]);
    }
    p.grp_begin[H] = (uint16_t)n;
    max_rows = gmax * t_q;
    if (max_rows > KVQ_MAX_ROWS) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

int tiles8_for(int rows) { return rows <= 8 ? 1 : rows <= 16 ? 2 : 4; }

struct Group {
    int b0, nb;          // sequences [b0, b0 + nb)
    int n_split, chunk;
    size_t ws_off;       // bytes
};

int round_up(long long x, int m) { return (int)((x + m - 1) / m * m); }

// Split policy: enough CTAs to fill every SM with whole waves.  Uniform lengths:
// the smallest split count (>= one wave) whose last wave is >= 90% full.
// Ragged lengths: a chunk of about a quarter wave's share of the positions.
// Chunks are multiples of gran (one stage per warp of the CTA) so that every
// warp gets the same number of stages; a chunk forced through KVQ_SPLIT only
// needs the 64-position segment alignment.
void choose_split(const kvq_cache *c, const Group &g, int max_len, int slots, int gran, int &n_split, int &chunk)
{
    const int H = c->n_kv_heads;
    long long total = 0;
    int lmax = 0, lmin = 0x7fffffff;
    for (int b = g.b0; b < g.b0 + g.nb; ++b) {
        if (c->n_segs[b] == 0) {
            lmin = 0;
            continue;
        }
        const kvq_segment &sl = seg_of(c, b, c->n_segs[b] - 1);
        const int L = std::min(max_len, sl.pos0 + sl.len);
        const int Lcap = std::min(max_len, sl.pos0 + sl.cap);
        total += (long long)L * H;
        lmax = std::max(lmax, Lcap);
        lmin = std::min(lmin, L);
    }
    if (lmax <= 0) {
        n_split = 1;
        chunk = KVQ_SEG_ALIGN;
        return;
    }
    const char *env = std::getenv("KVQ_SPLIT");
    if (env && std::atoi(env) > 0) {
        chunk = round_up(std::atoi(env), KVQ_SEG_ALIGN);
    } else {
        const int pairs = g.nb * H;
        const int max_n = std::max(1, (lmax + 255) / 256);   // at least 256 positions per split
        int n = 1;
        if (lmin * 2 >= lmax || total == 0) {
            const int n_min = std::max(1, (slots + pairs - 1) / pairs);
            double best = -1.0;
            n = std::min(n_min, max_n);   // short contexts: as many splits as the 256-position floor allows
            for (int k = n_min; k <= 4 * n_min && k <= max_n; ++k) {
                const double waves = (double)pairs * k / slots;
                const double eff = waves / std::ceil(waves);
                if (eff > best + 1e-9) {
                    best = eff;
                    n = k;
                }
                if (eff >= 0.9) break;
            }
            n = std::min(std::max(n, 1), max_n);
        } else {
            const long long per_cta = std::max<long long>(256, total / std::max(1, 4 * slots));
            n = (int)std::min<long long>(max_n, (lmax + per_cta - 1) / per_cta);
        }
        chunk = round_up((lmax + n - 1) / n, gran);
    }
    n_split = (lmax + chunk - 1) / chunk;
    if (n_split > 1024) {
        chunk = round_up((lmax + 1023) / 1024, gran);
        n_split = (lmax + chunk - 1) / chunk;
    }
}

// Partition the batch into launch groups (<= 64 sequences and <= 64 segments).
void make_groups(const kvq_cache *c, std::vector<Group> &gs)
{
    int b = 0;
    while (b < c->n_seqs) {
        Group g{b, 0, 1, KVQ_SEG_ALIGN, 0};
        int segs = 0;
        while (b < c->n_seqs && g.nb < kMaxSeqsLaunch && segs + c->n_segs[b] <= kMaxSegsLaunch) {
            segs += c->n_segs[b];
            ++g.nb;
            ++b;
        }
        gs.push_back(g);
    }
}

void fill_segments(const kvq_cache *c, const Group &g, AttnParams &p)
{
    int n = 0;
    for (int i = 0; i < g.nb; ++i) {
        const int b = g.b0 + i;
        p.seq_seg0[i] = (uint8_t)n;
        p.seq_nseg[i] = (uint8_t)c->n_segs[b];
        for (int k = 0; k < c->n_segs[b]; ++k, ++n) {
            const kvq_segment &s = seg_of(c, b, k);
            p.seg[n].kq = static_cast<const uint8_t *>(s.k_q);
            p.seg[n].ks = static_cast<const uint16_t *>(s.k_s);
            p.seg[n].vq = static_cast<const uint8_t *>(s.v_q);
            p.seg[n].vs = static_cast<const uint16_t *>(s.v_s);
            p.seg[n].pos0 = s.pos0;
            p.seg[n].cap = s.cap;
        }
    }
}

struct DecodeArgs {
    const kvq_cache *c;
    const void *q16;
    int n_q_heads, t_q, causal;
    const int32_t *seq_lens;
    int max_len;
    const int32_t *head_map;
    float sm_scale;
    float *out, *lse;
    void *workspace;
    size_t workspace_bytes;
    size_t *size_out;    // size query only: store the required workspace and return
    int8_t *dbg_qc;
    uint16_t *dbg_qs;
    int32_t *dbg_scores;
    bool dump;
    cudaStream_t stream;
};

kvq_status run_decode(const DecodeArgs &a)
{
    const kvq_cache *c = a.c;
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (a.t_q < 1 || a.t_q > KVQ_MAX_T_Q || a.max_len < 0) return KVQ_ERR_INVALID_ARG;
    if (!(std::isfinite(a.sm_scale))) return KVQ_ERR_INVALID_ARG;
    static thread_local AttnParams p;   // ~4 KB; kept off the stack
    std::memset(&p, 0, sizeof(p));
    int max_rows = 0;
    st = build_groups(c, a.n_q_heads, a.head_map, a.t_q, p, max_rows);
    if (st != KVQ_OK) return st;
    if (c->n_seqs == 0) {
        if (a.size_out) *a.size_out = 0;
        return KVQ_OK;
    }
    if (!a.size_out) {
        if (!a.q16 || !aligned16(a.q16) || !a.seq_lens) return KVQ_ERR_INVALID_ARG;
        if (a.dump ? (!a.dbg_qc || !a.dbg_qs || !a.dbg_scores) : (!a.out || !a.lse)) return KVQ_ERR_INVALID_ARG;
        if (!a.dump && (!aligned16(a.out) || (reinterpret_cast<uintptr_t>(a.lse) & 3u))) return KVQ_ERR_INVALID_ARG;
    }

    DeviceInfo *dev = nullptr;
    st = device_setup(&dev);
    if (st != KVQ_OK) return st;
    const int nt = tiles8_for(max_rows);
    const int slots = std::max(1, dev->n_sms * std::max(1, dev->ctas[c->v_type][nt]));

    std::vector<Group> gs;
    make_groups(c, gs);
    size_t ws = 0;
    const size_t rows_per_seq = (size_t)a.t_q * a.n_q_heads;
    for (Group &g : gs) {
        choose_split(c, g, a.max_len, slots, split_warps(nt) * kWTile, g.n_split, g.chunk);
        if (g.n_split > 1 && !a.dump) {
            g.ws_off = ws;
            const size_t bytes = (size_t)g.nb * rows_per_seq * g.n_split * (kD + 1) * sizeof(float);
            ws += (bytes + 255) / 256 * 256;
        }
    }
    if (a.size_out) {
        *a.size_out = ws;
        return KVQ_OK;
    }
    if (!a.dump && ws) {
        if (!a.workspace || a.workspace_bytes < ws || (reinterpret_cast<uintptr_t>(a.workspace) & 255u))
            return KVQ_ERR_WORKSPACE;
    }

    const bool pdl = pdl_enabled();
    const uint16_t *q = static_cast<const uint16_t *>(a.q16);
    for (const Group &g : gs) {
        fill_segments(c, g, p);
        const size_t r0 = (size_t)g.b0 * rows_per_seq;
        p.q = q + r0 * kD;
        p.seq_lens = a.seq_lens + g.b0;
        p.n_seqs = g.nb;
        p.n_kv_heads = c->n_kv_heads;
        p.n_q_heads = a.n_q_heads;
        p.t_q = a.t_q;
        p.causal = a.causal ? 1 : 0;
        p.max_len = a.max_len;
        p.n_split = g.n_split;
        p.chunk = g.chunk;
        p.qk_scale_log2 = a.sm_scale * 1.4426950408889634f;
        p.timeouts = dev->timeouts;
        if (a.dump) {
            p.dbg_qc = a.dbg_qc + r0 * kD;
            p.dbg_qs = a.dbg_qs + r0 * kNB;
            p.dbg_scores = a.dbg_scores + r0 * (size_t)a.max_len * kNB;
            p.out = nullptr;
            p.lse = nullptr;
            p.ws_o = p.ws_lse = nullptr;
        } else {
            p.dbg_qc = nullptr;
            p.dbg_qs = nullptr;
            p.dbg_scores = nullptr;
            p.out = a.out + r0 * kD;
            p.lse = a.lse + r0;
            if (g.n_split > 1) {
                char *w = static_cast<char *>(a.workspace) + g.ws_off;
                p.ws_o = reinterpret_cast<float *>(w);
                p.ws_lse = p.ws_o + (size_t)g.nb * rows_per_seq * g.n_split * kD;
            } else {
                p.ws_o = p.ws_lse = nullptr;
            }
        }
        cudaError_t e = (c->v_type == KVQ_V_Q4_0) ? launch_split_q4(p, nt, a.dump, a.stream, pdl)
                                                  : launch_split_q8(p, nt, a.dump, a.stream, pdl);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
        if (!a.dump && g.n_split > 1) {
            CombineParams cp;
            cp.ws_o = p.ws_o;
            cp.ws_lse = p.ws_lse;
            cp.out = p.out;
            cp.lse = p.lse;
            cp.n_rows = (int)(g.nb * rows_per_seq);
            cp.n_split = g.n_split;
            e = launch_combine(cp, a.stream, pdl);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return KVQ_ERR_CUDA;
            }
        }
    }
    return KVQ_OK;
}

}  // namespace

extern "C" {

const char *kvq_status_string(kvq_status s)
{
    switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported device or size";
    case KVQ_ERR_CAPACITY: return "segment capacity exceeded";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_TIMEOUT: return "a kernel wait gave up";
    }
    return "unknown status";
}

kvq_status kvq_append(kvq_cache *c, int32_t n_seqs_in, const int32_t *seq_ids, const int32_t *n_new,
                      const void *k16, const void *v16, void *stream)
{
    kvq_status st = check_cache(c);
    if (st != KVQ_OK) return st;
    if (n_seqs_in < 0) return KVQ_ERR_INVALID_ARG;
    if (n_seqs_in == 0) return KVQ_OK;
    if (!seq_ids || !n_new) return KVQ_ERR_INVALID_ARG;
    long long total = 0;
    std::vector<char> seen(c->n_seqs, 0);
    for (int i = 0; i < n_seqs_in; ++i) {
        const int b = seq_ids[i];
        if (b < 0 || b >= c->n_seqs || seen[b] || n_new[i] < 0) return KVQ_ERR_INVALID_ARG;
        if (n_new[i] > 0 && c->n_segs[b] < 1) return KVQ_ERR_INVALID_ARG;   // no open segment
        seen[b] = 1;
        total += n_new[i];
    }
    if (total == 0) return KVQ_OK;
    if (total > 0x7fffffffLL / c->n_kv_heads) return KVQ_ERR_INVALID_ARG;
    if (!k16 || !v16 || !aligned16(k16) || !aligned16(v16)) return KVQ_ERR_INVALID_ARG;
    for (int i = 0; i < n_seqs_in; ++i) {
        if (n_new[i] == 0) continue;
        const kvq_segment &s = seg_of(c, seq_ids[i], c->n_segs[seq_ids[i]] - 1);
        if ((long long)s.len + n_new[i] > s.cap) return KVQ_ERR_CAPACITY;
    }
    DeviceInfo *dev = nullptr;
    st = device_setup(&dev);
    if (st != KVQ_OK) return st;

    static thread_local AppendParams p;
    const bool pdl = pdl_enabled();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int src = 0, i = 0;
    while (i < n_seqs_in) {
        std::memset(&p, 0, sizeof(p));
        p.k16 = static_cast<const uint16_t *>(k16);
        p.v16 = static_cast<const uint16_t *>(v16);
        p.n_kv_heads = c->n_kv_heads;
        int max_rows = 0;
        while (i < n_seqs_in && p.n_entries < kMaxSeqsLaunch) {
            if (n_new[i] > 0) {
                const kvq_segment &sg = seg_of(c, seq_ids[i], c->n_segs[seq_ids[i]] - 1);
                AppendEntry &e = p.e[p.n_entries++];
                e.kq = static_cast<uint8_t *>(sg.k_q);
                e.ks = static_cast<uint16_t *>(sg.k_s);
                e.vq = static_cast<uint8_t *>(sg.v_q);
                e.vs = static_cast<uint16_t *>(sg.v_s);
                e.cap = sg.cap;
                e.dst = sg.len;
                e.src = src;
                e.n = n_new[i];
                max_rows = std::max(max_rows, n_new[i] * c->n_kv_heads);
            }
            src += n_new[i];
            ++i;
        }
        if (p.n_entries == 0) continue;
        if (launch_append(p, c->v_type, max_rows, s, pdl) != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
    }
    for (int j = 0; j < n_seqs_in; ++j)
        if (n_new[j] > 0) c->segs[(size_t)seq_ids[j] * c->max_segs + c->n_segs[seq_ids[j]] - 1].len += n_new[j];
    return KVQ_OK;
}

kvq_status kvq_decode_attn(const kvq_cache *c, const void *q16, int32_t n_q_heads, int32_t t_q,
                           int32_t causal_tail, const int32_t *seq_lens, int32_t max_len,
                           const int32_t *head_map, float sm_scale, float *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    DecodeArgs a{};
    a.c = c;
    a.q16 = q16;
    a.n_q_heads = n_q_heads;
    a.t_q = t_q;
    a.causal = causal_tail;
    a.seq_lens = seq_lens;
    a.max_len = max_len;
    a.head_map = head_map;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.dump = false;
    a.stream = static_cast<cudaStream_t>(stream);
    return run_decode(a);
}

kvq_status kvq_decode_workspace_size(const kvq_cache *c, int32_t n_q_heads, int32_t t_q, int32_t max_len,
                                     const int32_t *head_map, size_t *bytes)
{
    if (!bytes) return KVQ_ERR_INVALID_ARG;
    DecodeArgs a{};
    a.c = c;
    a.n_q_heads = n_q_heads;
    a.t_q = t_q;
    a.max_len = max_len;
    a.head_map = head_map;
    a.sm_scale = 1.0f;
    a.size_out = bytes;
    return run_decode(a);
}

kvq_status kvq_debug_qk(const kvq_cache *c, const void *q16, int32_t n_q_heads, int32_t t_q,
                        const int32_t *seq_lens, int32_t max_len, const int32_t *head_map, int8_t *q_codes,
                        uint16_t *q_scales, int32_t *scores, void *stream)
{
    DecodeArgs a{};
    a.c = c;
    a.q16 = q16;
    a.n_q_heads = n_q_heads;
    a.t_q = t_q;
    a.causal = 0;
    a.seq_lens = seq_lens;
    a.max_len = max_len;
    a.head_map = head_map;
    a.sm_scale = 1.0f;
    a.dbg_qc = q_codes;
    a.dbg_qs = q_scales;
    a.dbg_scores = scores;
    a.dump = true;
    a.stream = static_cast<cudaStream_t>(stream);
    return run_decode(a);
}

}  // extern "C"

// Scratch of kvq_decode_attn_noalloc: a file-scope device array, so callers
// that cannot allocate never need to pass a workspace.  Host code must not use
// the symbol itself as a pointer; its device address is looked up once per
// device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up once).
kvq_status noalloc_scratch(void **ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KVQ_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return KVQ_OK;
}
}  // namespace

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_cache *c, const void *q16, int32_t n_q_heads, int32_t t_q,
                                              int32_t causal_tail, const int32_t *seq_lens, int32_t max_len,
                                              const int32_t *head_map, float sm_scale, float *out, float *lse,
                                              void *stream)
{
    kvq_status st = check_cache(c);   // reject bad descriptors before touching the device
    if (st != KVQ_OK) return st;
    DeviceInfo *dev = nullptr;
    st = device_setup(&dev);
    if (st != KVQ_OK) return st;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != KVQ_OK) return st;
    return kvq_decode_attn(c, q16, n_q_heads, t_q, causal_tail, seq_lens, max_len, head_map, sm_scale, out, lse,
                           scratch, KVQ_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" kvq_status kvq_wait_timeouts(uint32_t *count)
{
    if (!count) return KVQ_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    kvq_status st = device_setup(&dev);
    if (st != KVQ_OK) return st;
    unsigned int n = 0;
    if (cudaMemcpy(&n, dev->timeouts, sizeof(n), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return KVQ_ERR_CUDA;
    }
    *count = n;
    return n ? KVQ_ERR_TIMEOUT : KVQ_OK;
}
