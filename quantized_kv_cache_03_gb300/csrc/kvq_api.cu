// kvq_api.cu -- the C ABI of libkvq.so: argument validation, segment-table
// marshalling, split policy and kernel launches.  No allocation, and no host
// sync except in kvq_wait_timeouts.
#include <climits>
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
    int ctas[2][2][5] = {};   // [k_type][v_type][n_tiles8] resident split CTAs per SM
    int ctas_half[2][2] = {};   // [k_type][v_type] the same for the 8-row kernel with kWarpsHalf warps
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
            const int w = split_warps(nt);
            if (prepare_split_q4(nt, w, KVQ_K_I8, kModeDecode, &d.ctas[KVQ_K_I8][KVQ_V_Q4_0][nt]) != cudaSuccess ||
                prepare_split_q8(nt, w, KVQ_K_I8, kModeDecode, &d.ctas[KVQ_K_I8][KVQ_V_Q8_0][nt]) != cudaSuccess ||
                prepare_split_q4(nt, w, KVQ_K_F16, kModeDecode, &d.ctas[KVQ_K_F16][KVQ_V_Q4_0][nt]) != cudaSuccess ||
                prepare_split_q8(nt, w, KVQ_K_F16, kModeDecode, &d.ctas[KVQ_K_F16][KVQ_V_Q8_0][nt]) != cudaSuccess ||
                prepare_split_q4(nt, w, KVQ_K_I8, kModeDump, nullptr) != cudaSuccess ||
                prepare_split_q8(nt, w, KVQ_K_I8, kModeDump, nullptr) != cudaSuccess) {
                cudaGetLastError();
                return KVQ_ERR_CUDA;
            }
        }
        if (prepare_split_q4(1, kWarpsHalf, KVQ_K_I8, kModeDecode, &d.ctas_half[KVQ_K_I8][KVQ_V_Q4_0]) != cudaSuccess ||
            prepare_split_q8(1, kWarpsHalf, KVQ_K_I8, kModeDecode, &d.ctas_half[KVQ_K_I8][KVQ_V_Q8_0]) != cudaSuccess ||
            prepare_split_q4(1, kWarpsHalf, KVQ_K_F16, kModeDecode, &d.ctas_half[KVQ_K_F16][KVQ_V_Q4_0]) != cudaSuccess ||
            prepare_split_q8(1, kWarpsHalf, KVQ_K_F16, kModeDecode, &d.ctas_half[KVQ_K_F16][KVQ_V_Q8_0]) != cudaSuccess ||
            prepare_split_q4(1, split_warps(1), KVQ_K_I8, kModeLoseStage, nullptr) != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
        if (prepare_prefill_q4() != cudaSuccess || prepare_prefill_q8() != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
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
    if (c->k_type != KVQ_K_I8 && c->k_type != KVQ_K_F16) return KVQ_ERR_INVALID_ARG;
    const bool f16k = c->k_type == KVQ_K_F16;   // no K scales
    if (c->head_dim != KVQ_HEAD_DIM) return c->head_dim % KVQ_QBLOCK ? KVQ_ERR_INVALID_ARG : KVQ_ERR_UNSUPPORTED;
    if (c->n_seqs == 0) return KVQ_OK;
    if (!c->n_segs || !c->segs) return KVQ_ERR_INVALID_ARG;
    for (int b = 0; b < c->n_seqs; ++b) {
        const int ns = c->n_segs[b];
        if (ns < 0 || ns > c->max_segs || ns > kMaxSegsLaunch) return KVQ_ERR_INVALID_ARG;
        for (int k = 0; k < ns; ++k) {
            const kvq_segment &s = seg_of(c, b, k);
            if (!s.k_q || (!s.k_s && !f16k) || !s.v_q || !s.v_s) return KVQ_ERR_INVALID_ARG;
            if (!aligned16(s.k_q) || !aligned16(s.k_s) || !aligned16(s.v_q) || !aligned16(s.v_s))
                return KVQ_ERR_INVALID_ARG;
            if (s.cap <= 0 || s.cap % KVQ_SEG_ALIGN || s.len < 0 || s.len > s.cap) return KVQ_ERR_INVALID_ARG;
            if (s.layout != KVQ_LAYOUT_TILES && s.layout != KVQ_LAYOUT_ROWS) return KVQ_ERR_INVALID_ARG;
            if (s.layout == KVQ_LAYOUT_ROWS && f16k) return KVQ_ERR_UNSUPPORTED;   // rows layout: int8 K only
            const long long expect = k == 0 ? 0 : (long long)seg_of(c, b, k - 1).pos0 + seg_of(c, b, k - 1).len;
            if (s.pos0 != expect) return KVQ_ERR_INVALID_ARG;
            if ((long long)s.pos0 + s.cap > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;
        }
    }
    return KVQ_OK;
}

// One decode call (one cache) as the planner sees it.
struct Desc {
    const kvq_cache *c;
    const uint16_t *q;
    int n_q_heads, t_q, causal;
    const int32_t *seq_lens;
    int max_len;
    float sm_scale;
    float *out, *lse;
    int8_t *dbg_qc;
    uint16_t *dbg_qs;
    int32_t *dbg_scores;
    const uint16_t *k_new, *v_new;   // fused append of t_q tokens per sequence, or null
    std::vector<int> kv;   // query head -> kv head
    int max_rows;          // query rows of the busiest kv head
    bool has_rows;         // some segment of the cache keeps KVQ_LAYOUT_ROWS
};

// Validate one call's shape arguments and derive its head map.
kvq_status prepare_desc(Desc &d, const int32_t *head_map, bool need_ptrs, bool dump)
{
    kvq_status st = check_cache(d.c);
    if (st != KVQ_OK) return st;
    const kvq_cache *c = d.c;
    if (d.t_q < 1 || d.t_q > KVQ_MAX_T_Q || d.max_len < 0) return KVQ_ERR_INVALID_ARG;
    if (!(std::isfinite(d.sm_scale))) return KVQ_ERR_INVALID_ARG;
    const int H = c->n_kv_heads;
    if (d.n_q_heads < 1 || d.n_q_heads > KVQ_MAX_HEADS) return KVQ_ERR_INVALID_ARG;
    d.kv.assign(d.n_q_heads, 0);
    if (head_map) {
        for (int h = 0; h < d.n_q_heads; ++h) {
            if (head_map[h] < 0 || head_map[h] >= H) return KVQ_ERR_INVALID_ARG;
            d.kv[h] = head_map[h];
        }
    } else {
        if (d.n_q_heads % H) return KVQ_ERR_INVALID_ARG;
        const int gsz = d.n_q_heads / H;
        for (int h = 0; h < d.n_q_heads; ++h) d.kv[h] = h / gsz;
    }
    std::vector<int> cnt(H, 0);
    for (int h = 0; h < d.n_q_heads; ++h) ++cnt[d.kv[h]];
    int gmax = 0;
    for (int k = 0; k < H; ++k) gmax = std::max(gmax, cnt[k]);
    d.max_rows = gmax * d.t_q;   // at most 256 * 4096: row tiles of <= KVQ_MAX_ROWS
    d.has_rows = false;
    for (int b = 0; b < c->n_seqs; ++b)
        for (int k = 0; k < c->n_segs[b]; ++k) d.has_rows = d.has_rows || seg_of(c, b, k).layout == KVQ_LAYOUT_ROWS;
    // F16 K: no fused append and no integer-score dump
    if (c->k_type == KVQ_K_F16 && (dump || d.k_new || d.v_new)) return KVQ_ERR_UNSUPPORTED;
    if ((d.k_new != nullptr) != (d.v_new != nullptr)) return KVQ_ERR_INVALID_ARG;
    if (d.k_new) {
        if (dump || !aligned16(d.k_new) || !aligned16(d.v_new)) return KVQ_ERR_INVALID_ARG;
        if (d.t_q > KVQ_MAX_T_Q_APPEND) return KVQ_ERR_UNSUPPORTED;
        for (int b = 0; b < c->n_seqs; ++b) {
            if (c->n_segs[b] < 1) return KVQ_ERR_INVALID_ARG;   // no open segment
            const kvq_segment &sl = seg_of(c, b, c->n_segs[b] - 1);
            if ((long long)sl.len + d.t_q > sl.cap) return KVQ_ERR_CAPACITY;
        }
    }
    if (need_ptrs && c->n_seqs > 0) {
        if (!d.q || !aligned16(d.q) || !d.seq_lens) return KVQ_ERR_INVALID_ARG;
        if (dump ? (!d.dbg_qc || !d.dbg_qs || !d.dbg_scores) : (!d.out || !d.lse)) return KVQ_ERR_INVALID_ARG;
        if (!dump && (!aligned16(d.out) || (reinterpret_cast<uintptr_t>(d.lse) & 3u))) return KVQ_ERR_INVALID_ARG;
    }
    return KVQ_OK;
}

// 8-row tiles per CTA of the split kernel for a call with `rows` query rows per
// kv head: 1, 2 or 4.  KVQ_ROW_TILE=16 caps calls with more than 16 rows at
// the 16-row kernel (the kv head's rows are then taken by several row-tile
// CTAs that stream the same positions); the 8-row kernel has no row tiles.
int tiles8_for(int rows)
{
    const char *e = std::getenv("KVQ_ROW_TILE");
    const int cap = (e && std::atoi(e) == 16) ? 2 : 4;
    return std::min(cap, rows <= 8 ? 1 : rows <= 16 ? 2 : 4);
}


// Query rows per kv head from which a call runs on the tcgen05 kernel (one CTA
// per 128-row tile; a tile with fewer rows leaves the softmax warps of its
// empty TMEM lane quarters idle): chunks of more than 32 rows.  The verify
// shape (32 rows per kv head) measured 1007 us there against 520 us on the
// split kernel's 32-row tiles: the tcgen05 kernel's per-tile period is set by
// one lane quarter's softmax latency, which 32 rows do not shorten.
// KVQ_TC_ROWS=<rows> moves the threshold; KVQ_PREFILL=0 keeps every call on
// the split kernel.
constexpr int kTcMinRows = KVQ_MAX_ROWS + 1;
int tc_min_rows()
{
    const char *e = std::getenv("KVQ_TC_ROWS");
    return (e && std::atoi(e) > 0) ? std::atoi(e) : kTcMinRows;
}
// The tcgen05 kernel reads tile-layout segments only (caches holding a
// rows-layout segment take the split kernel's row tiles) and has no fused
// append (a call carrying its step's tokens gets an append launch first).  The
// score dump takes the same route, so it tests the kernel the decode call runs.
bool tc_rows(const Desc &d)
{
    const char *e = std::getenv("KVQ_PREFILL");
    const bool on = !(e && e[0] == '0');
    return on && !d.has_rows && d.c->k_type == KVQ_K_I8 && d.max_rows >= tc_min_rows();
}
bool prefill_kernel_for(const Desc &d) { return !d.k_new && tc_rows(d); }

// The step's tokens of call d (t_q per sequence, token-major as kvq_append
// takes them) through the append kernel, for a call whose attention runs on
// the tcgen05 kernel.  The caller bumps the host lengths.
cudaError_t launch_step_append(const Desc &d, cudaStream_t s, bool pdl)
{
    static thread_local AppendParams p;
    const kvq_cache *c = d.c;
    int b = 0;
    while (b < c->n_seqs) {
        std::memset(&p, 0, sizeof(p));
        p.k16 = d.k_new;
        p.v16 = d.v_new;
        p.n_kv_heads = c->n_kv_heads;
        while (b < c->n_seqs && p.n_entries < kMaxSeqsLaunch) {
            const kvq_segment &sg = seg_of(c, b, c->n_segs[b] - 1);
            AppendEntry &e = p.e[p.n_entries++];
            e.kq = static_cast<uint8_t *>(sg.k_q);
            e.ks = static_cast<uint16_t *>(sg.k_s);
            e.vq = static_cast<uint8_t *>(sg.v_q);
            e.vs = static_cast<uint16_t *>(sg.v_s);
            e.cap = sg.cap;
            e.dst = sg.len;
            e.src = b * d.t_q;
            e.n = d.t_q;
            e.layout = sg.layout;
            ++b;
        }
        const cudaError_t err = launch_append(p, c->v_type, c->k_type, d.t_q * c->n_kv_heads, s, pdl);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// Calls whose rows go to the tcgen05 kernel take their step's tokens through
// an append launch first: dsp is ds with those calls' k_new / v_new cleared,
// pre their indices.
void split_off_pre_appends(const std::vector<Desc> &ds, std::vector<Desc> &dsp, std::vector<int> &pre)
{
    dsp = ds;
    pre.clear();
    for (size_t i = 0; i < ds.size(); ++i)
        if (ds[i].k_new && ds[i].c->n_seqs > 0 && tc_rows(ds[i])) {
            dsp[i].k_new = dsp[i].v_new = nullptr;
            pre.push_back((int)i);
        }
}
int round_up(long long x, int m) { return (int)((x + m - 1) / m * m); }

// Positions of sequence b that the kernel may visit: the end of its last
// segment's capacity, cut at max_len.
int seq_reach(const kvq_cache *c, int b, int max_len)
{
    if (c->n_segs[b] == 0) return 0;
    const kvq_segment &sl = seg_of(c, b, c->n_segs[b] - 1);
    return std::max(0, std::min(max_len, sl.pos0 + sl.cap));
}

// A work group: sequences [b0, b0 + nb) of call d.
struct Unit {
    int d, b0, nb;
    int reach;          // max seq_reach over the unit
    int n_rt;           // row tiles of 8 * NT query rows per kv head
    int n_split;
    size_t ws_off;      // bytes
    int cta0, row0;
};

// A split launch: units of calls with one V format and one kernel, run in one
// grid.  prefill: the tcgen05 kernel (128-row tiles) for calls with more query
// rows per kv head than the split kernel's 32-row tile and no fused append.
struct Launch {
    int v_type = 0, k_type = 0, nt = 1;
    int warps = 0;   // warps per split CTA (split_warps(nt), or kWarpsHalf for the 8-row kernel)
    bool prefill = false;
    int chunk = KVQ_SEG_ALIGN;
    int chunk0 = KVQ_SEG_ALIGN;   // split 0's positions (chunk unless the launch is split unevenly)
    bool split_major = false;     // CTAs ordered split first (the uneven split's large pieces first)
    int n_ctas = 0, n_rows = 0;   // split CTAs, combine rows
    std::vector<Unit> units;
};

// Query rows one CTA of the launch takes per kv head.
int tile_rows(const Launch &ln) { return ln.prefill ? kPrefillRows : 8 * ln.nt; }

// Split policy, one chunk per launch so that CTAs of every unit do the same
// amount of work.  For a candidate chunk c the launch has n CTAs with work
// W (kv positions) in total; with `slots` CTAs resident at once and a fixed
// cost of about kOverhead positions per CTA, the finish time is estimated as
// c + overhead when one wave holds every CTA, else (W + n * overhead) / slots
// plus one more CTA for the tail.  The cheapest candidate wins (the larger
// chunk on ties).  Chunks are multiples of gran (one stage per warp of the
// CTA) and at least 256 positions; KVQ_SPLIT forces a chunk (rounded to the
// 64-position segment alignment).
constexpr int kOverhead = 512;
int choose_chunk(const std::vector<Desc> &ds, const Launch &ln, int slots, int gran)
{
    int lmax = 0;
    for (const Unit &u : ln.units) lmax = std::max(lmax, u.reach);
    if (lmax <= 0) return KVQ_SEG_ALIGN;
    const char *env = std::getenv("KVQ_SPLIT");
    int chunk;
    if (env && std::atoi(env) > 0) {
        chunk = round_up(std::atoi(env), KVQ_SEG_ALIGN);
    } else {
        std::vector<std::pair<int, int>> seqs;   // (kv heads x row tiles, reach)
        long long W = 0;
        for (const Unit &u : ln.units) {
            const kvq_cache *c = ds[u.d].c;
            const int n_rt = (ds[u.d].max_rows + tile_rows(ln) - 1) / tile_rows(ln);
            for (int b = u.b0; b < u.b0 + u.nb; ++b) {
                const int r = seq_reach(c, b, ds[u.d].max_len);
                seqs.push_back({c->n_kv_heads * n_rt, r});
                W += (long long)r * c->n_kv_heads * n_rt;
            }
        }
        const int max_n = std::max(1, std::min(1024, (lmax + 255) / 256));
        double best = 1e300;
        chunk = round_up(lmax, gran);
        int prev = -1;
        for (int n = 1; n <= max_n; n = (n < 128) ? n + 1 : n + n / 16) {
            const int cand = std::max(round_up(256, gran), round_up((lmax + n - 1) / n, gran));
            if (cand == prev) continue;
            prev = cand;
            long long ctas = 0;
            for (const auto &q : seqs) ctas += (long long)q.first * std::max(1, (q.second + cand - 1) / cand);
            const double cmax = std::min(cand, lmax) + kOverhead;
            const double est = ctas <= slots ? cmax : (double)(W + ctas * kOverhead) / slots + cmax;
            if (est < best - 1e-9) {
                best = est;
                chunk = cand;
            }
        }
    }
    if ((lmax + chunk - 1) / chunk > 1024) chunk = round_up((lmax + 1023) / 1024, gran);
    return chunk;
}

// Uneven two-way split of a one-wave tcgen05 launch.  With U CTAs of one
// group on S SMs (S / 2 < U < S; one CTA per SM), S - U SMs idle for the whole
// launch.  Splitting every unit at c0 instead gives U large CTAs [0, c0),
// dispatched first, and U small ones [c0, reach) that the S - U idle SMs take
// k = ceil(U / (S - U)) at a time; the combine merges the two partials.
// c0 balances the large CTAs' time c0 + o against k (reach - c0 + o), o the
// fixed cost of one CTA in positions (KVQ_PREFILL_CTA_COST overrides it).
// KVQ_PREFILL_BALANCE=0 turns the split off, a positive value forces k.  A
// chunk forced by KVQ_SPLIT keeps even splits.  Returns false (launch
// unchanged) when the split does not pay by at least 5 %.
constexpr int kPrefillCtaCost = 256;
bool uneven_split(const std::vector<Desc> &ds, Launch &ln, int n_sms)
{
    if (!ln.prefill || ln.units.size() != 1) return false;
    const char *fs = std::getenv("KVQ_SPLIT");
    if (fs && std::atoi(fs) > 0) return false;
    const char *env = std::getenv("KVQ_PREFILL_BALANCE");
    const int forced = env ? std::atoi(env) : -1;
    if (forced == 0) return false;
    const Unit &u = ln.units[0];
    const Desc &d = ds[u.d];
    const int lmax = u.reach;
    if (lmax <= 0 || ln.chunk < lmax) return false;   // already split evenly
    const long long U = (long long)((d.max_rows + kPrefillRows - 1) / kPrefillRows) * d.c->n_kv_heads * u.nb;
    if (U >= n_sms || 2 * U <= n_sms) return false;
    const long long k = forced > 0 ? forced : (U + (n_sms - U) - 1) / (n_sms - U);
    const char *ce = std::getenv("KVQ_PREFILL_CTA_COST");
    const long long o = (ce && std::atoi(ce) >= 0) ? std::atoi(ce) : kPrefillCtaCost;
    const int c0 = round_up((int)((k * lmax + (k - 1) * o + k) / (k + 1)), kPrefillPositions);
    if (c0 >= lmax || (double)(c0 + o) > 0.95 * (double)(lmax + o)) return false;
    ln.chunk0 = c0;
    ln.chunk = round_up(lmax - c0, kPrefillPositions);
    ln.split_major = true;
    return true;
}

// Pack the calls' sequences into launches (tables of AttnParams bound the
// segments, sequences, groups and head-table entries of one launch).
kvq_status plan(std::vector<Desc> &ds, DeviceInfo *dev, bool dump, std::vector<Launch> &out, size_t &ws)
{
    out.clear();
    ws = 0;
    Launch cur;
    int segs = 0, seqs = 0, heads = 0, kvs = 0, last_d = -1;
    auto flush = [&]() {
        if (!cur.units.empty()) out.push_back(cur);
        cur = Launch();
        segs = seqs = heads = kvs = 0;
        last_d = -1;
    };
    for (int di = 0; di < (int)ds.size(); ++di) {
        const kvq_cache *c = ds[di].c;
        if (c->n_seqs == 0) continue;
        const bool pf = prefill_kernel_for(ds[di]);
        if (!cur.units.empty() && (cur.v_type != c->v_type || cur.k_type != c->k_type || cur.prefill != pf))
            flush();
        int b = 0;
        while (b < c->n_seqs) {
            const bool new_desc = last_d != di;
            const int need_heads = new_desc ? ds[di].n_q_heads : 0, need_kv = new_desc ? c->n_kv_heads + 1 : 0;
            if (cur.units.size() == (size_t)kMaxGroups || seqs == kMaxSeqsLaunch ||
                segs + c->n_segs[b] > kMaxSegsLaunch || heads + need_heads > kMaxHeadTab ||
                kvs + need_kv > kMaxHeadTab + kMaxGroups) {
                flush();
                continue;
            }
            if (cur.units.empty()) {
                cur.v_type = c->v_type;
                cur.k_type = c->k_type;
                cur.prefill = pf;
            }
            heads += need_heads;
            kvs += need_kv;
            last_d = di;
            Unit u{di, b, 0, 0, 1, 1, 0, 0, 0};
            while (b < c->n_seqs && seqs < kMaxSeqsLaunch && segs + c->n_segs[b] <= kMaxSegsLaunch) {
                segs += c->n_segs[b];
                u.reach = std::max(u.reach, seq_reach(c, b, ds[di].max_len));
                ++seqs;
                ++u.nb;
                ++b;
            }
            cur.nt = std::max(cur.nt, tiles8_for(std::min(ds[di].max_rows, KVQ_MAX_ROWS)));
            cur.units.push_back(u);
        }
    }
    flush();
    for (Launch &ln : out) {
        const bool tc = ln.prefill;   // the tcgen05 kernel: one CTA per SM
        const int slots = tc ? dev->n_sms : std::max(1, dev->n_sms * std::max(1, dev->ctas[ln.k_type][ln.v_type][ln.nt]));
        ln.warps = tc ? 0 : split_warps(ln.nt);
        ln.chunk = choose_chunk(ds, ln, slots, ln.prefill ? kPrefillPositions : ln.warps * kWTile);
        // The 8-row kernel with half the warps (two CTAs per SM) when the full
        // CTAs take more than one wave; KVQ_SPLIT_WARPS=8 or 16 forces either.
        // A chunk forced by KVQ_SPLIT keeps the full CTAs unless asked, so that
        // one forced chunk gives one partition of the positions.
        const int half_ctas = dev->ctas_half[ln.k_type][ln.v_type];
        if (!tc && ln.nt == 1 && !dump && half_ctas >= 2) {
            const char *e = std::getenv("KVQ_SPLIT_WARPS");
            const char *fs = std::getenv("KVQ_SPLIT");
            const int force = e ? std::atoi(e) : 0;
            bool half = force == kWarpsHalf;
            if (force != kWarpsHalf && force != split_warps(1) && !(fs && std::atoi(fs) > 0)) {
                long long n = 0;
                for (const Unit &u : ln.units)
                    n += (long long)std::max(1, (u.reach + ln.chunk - 1) / ln.chunk) * ds[u.d].c->n_kv_heads * u.nb;
                half = n > slots;
            }
            if (half) {
                ln.warps = kWarpsHalf;
                ln.chunk = choose_chunk(ds, ln, dev->n_sms * half_ctas, kWarpsHalf * kWTile);
            }
        }
        ln.chunk0 = ln.chunk;
        if (tc) uneven_split(ds, ln, dev->n_sms);
        for (Unit &u : ln.units) {
            const Desc &d = ds[u.d];
            u.n_split = u.reach <= ln.chunk0 ? 1 : 1 + (u.reach - ln.chunk0 + ln.chunk - 1) / ln.chunk;
            u.n_rt = (d.max_rows + tile_rows(ln) - 1) / tile_rows(ln);   // 1 unless rows exceed the tile
            const long long n = (long long)u.n_rt * u.n_split * d.c->n_kv_heads * u.nb;
            if (ln.n_ctas + n > INT_MAX) return KVQ_ERR_UNSUPPORTED;
            u.cta0 = ln.n_ctas;
            ln.n_ctas += (int)n;
            if (u.n_split > 1 && !dump) {
                const size_t rows = (size_t)u.nb * d.t_q * d.n_q_heads;
                u.row0 = ln.n_rows;
                ln.n_rows += (int)rows;
                u.ws_off = ws;
                ws += (rows * u.n_split * (kD + 1) * sizeof(float) + 255) / 256 * 256;
            }
        }
    }
    return KVQ_OK;
}

void fill_launch(const std::vector<Desc> &ds, const Launch &ln, bool dump, void *workspace, unsigned int *timeouts,
                 AttnParams &p, CombineParams &cp)
{
    std::memset(&p, 0, sizeof(p));
    std::memset(&cp, 0, sizeof(cp));
    int nseg = 0, nseq = 0, nhead = 0, nkv = 0, last_d = -1, head0 = 0;
    for (const Unit &u : ln.units) {
        const Desc &d = ds[u.d];
        const kvq_cache *c = d.c;
        if (u.d != last_d) {   // this call's head table
            head0 = nkv;
            for (int k = 0; k < c->n_kv_heads; ++k) {
                p.grp_begin[nkv++] = (uint16_t)nhead;
                for (int h = 0; h < d.n_q_heads; ++h)
                    if (d.kv[h] == k) p.grp_q[nhead++] = (uint16_t)h;
            }
            p.grp_begin[nkv++] = (uint16_t)nhead;
            last_d = u.d;
        }
        GroupDesc &G = p.grp[p.n_groups];
        const size_t rows_per_seq = (size_t)d.t_q * d.n_q_heads;
        const size_t r0 = (size_t)u.b0 * rows_per_seq;
        G.q = d.q ? d.q + r0 * kD : nullptr;
        if (d.k_new) {
            const size_t t0 = (size_t)u.b0 * d.t_q * c->n_kv_heads * kD;
            G.k_new = d.k_new + t0;
            G.v_new = d.v_new + t0;
        }
        G.seq_lens = d.seq_lens ? d.seq_lens + u.b0 : nullptr;
        G.cta0 = u.cta0;
        G.seq0 = nseq;
        G.head0 = head0;
        G.n_seqs = u.nb;
        G.n_kv_heads = c->n_kv_heads;
        G.n_q_heads = d.n_q_heads;
        G.t_q = d.t_q;
        G.causal = d.causal ? 1 : 0;
        G.max_len = d.max_len;
        G.n_split = u.n_split;
        G.n_rt = u.n_rt;
        G.chunk = ln.chunk;
        G.chunk0 = ln.chunk0;
        G.split_major = ln.split_major ? 1 : 0;
        G.qk_scale_log2 = d.sm_scale * 1.4426950408889634f;
        if (dump) {
            G.dbg_qc = d.dbg_qc + r0 * kD;
            G.dbg_qs = d.dbg_qs + r0 * kNB;
            G.dbg_scores = d.dbg_scores + r0 * (size_t)d.max_len * kNB;
        } else {
            G.out = d.out + r0 * kD;
            G.lse = d.lse + r0;
            if (u.n_split > 1) {
                char *w = static_cast<char *>(workspace) + u.ws_off;
                G.ws_o = reinterpret_cast<float *>(w);
                G.ws_lse = G.ws_o + (size_t)u.nb * rows_per_seq * u.n_split * kD;
                CombineGroup &cg = cp.grp[cp.n_groups++];
                cg.ws_o = G.ws_o;
                cg.ws_lse = G.ws_lse;
                cg.out = G.out;
                cg.lse = G.lse;
                cg.row0 = u.row0;
                cg.n_split = u.n_split;
            }
        }
        ++p.n_groups;
        for (int i = 0; i < u.nb; ++i) {
            const int b = u.b0 + i;
            p.seq_seg0[nseq] = (uint8_t)nseg;
            p.seq_nseg[nseq] = (uint8_t)c->n_segs[b];
            if (c->n_segs[b] > 0) {
                const kvq_segment &sl = seg_of(c, b, c->n_segs[b] - 1);
                p.app_pos[nseq] = sl.pos0 + sl.len;
            }
            ++nseq;
            for (int k = 0; k < c->n_segs[b]; ++k, ++nseg) {
                const kvq_segment &s = seg_of(c, b, k);
                p.seg[nseg].kq = static_cast<const uint8_t *>(s.k_q);
                p.seg[nseg].ks = static_cast<const uint16_t *>(s.k_s);
                p.seg[nseg].vq = static_cast<const uint8_t *>(s.v_q);
                p.seg[nseg].vs = static_cast<const uint16_t *>(s.v_s);
                p.seg[nseg].pos0 = s.pos0;
                p.seg[nseg].cap = s.cap;
                p.seg[nseg].layout = s.layout;
            }
        }
    }
    p.timeouts = timeouts;
}

// Plan, check the workspace and launch (or, with size_out, only report the
// workspace the calls need).
kvq_status run(std::vector<Desc> &ds, bool dump, void *workspace, size_t workspace_bytes, size_t *size_out,
               cudaStream_t stream, int32_t *kernel_out = nullptr, bool lose_stage = false)
{
    DeviceInfo *dev = nullptr;
    bool any = false;
    for (const Desc &d : ds) any = any || d.c->n_seqs > 0;
    if (!any) {
        if (size_out) *size_out = 0;
        return KVQ_OK;
    }
    kvq_status st = device_setup(&dev);
    if (st != KVQ_OK) return st;
    std::vector<Desc> dsp;
    std::vector<int> pre;
    split_off_pre_appends(ds, dsp, pre);
    std::vector<Launch> lns;
    size_t ws = 0;
    st = plan(dsp, dev, dump, lns, ws);
    if (st != KVQ_OK) return st;
    if (kernel_out) *kernel_out = (!lns.empty() && lns[0].prefill) ? 1 : 0;
    if (lose_stage)   // the test flavour exists for one form of the split kernel
        for (const Launch &ln : lns)
            if (ln.prefill || ln.nt != 1 || ln.warps != split_warps(1) || ln.k_type != KVQ_K_I8 ||
                ln.v_type != KVQ_V_Q4_0)
                return KVQ_ERR_UNSUPPORTED;
    const int mode = dump ? kModeDump : lose_stage ? kModeLoseStage : kModeDecode;
    if (size_out) {
        *size_out = ws;
        return KVQ_OK;
    }
    if (!dump && ws) {
        if (!workspace || workspace_bytes < ws || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return KVQ_ERR_WORKSPACE;
    }
    static thread_local AttnParams p;        // ~6 KB; kept off the stack
    static thread_local CombineParams cp;
    const bool pdl = pdl_enabled();
    for (int i : pre)
        if (launch_step_append(ds[i], stream, pdl) != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
    for (const Launch &ln : lns) {
        fill_launch(dsp, ln, dump, workspace, dev->timeouts, p, cp);
        cudaError_t e;
        if (ln.prefill)
            e = (ln.v_type == KVQ_V_Q4_0) ? launch_prefill_q4(p, ln.n_ctas, dump, stream, pdl)
                                          : launch_prefill_q8(p, ln.n_ctas, dump, stream, pdl);
        else
            e = (ln.v_type == KVQ_V_Q4_0) ? launch_split_q4(p, ln.nt, ln.warps, ln.k_type, ln.n_ctas, mode, stream, pdl)
                                          : launch_split_q8(p, ln.nt, ln.warps, ln.k_type, ln.n_ctas, mode, stream, pdl);
        if (e == cudaSuccess && ln.n_rows > 0) e = launch_combine(cp, ln.n_rows, stream, pdl);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return KVQ_ERR_CUDA;
        }
    }
    for (const Desc &d : ds)   // fused appends: the open segments grew
        if (d.k_new)
            for (int b = 0; b < d.c->n_seqs; ++b)
                const_cast<kvq_cache *>(d.c)->segs[(size_t)b * d.c->max_segs + d.c->n_segs[b] - 1].len += d.t_q;
    return KVQ_OK;
}

// kvq_decode_desc (public) -> Desc, validated.
kvq_status to_desc(const kvq_decode_desc &x, bool need_ptrs, Desc &d)
{
    d = Desc();
    d.c = x.cache;
    d.q = static_cast<const uint16_t *>(x.q16);
    d.n_q_heads = x.n_q_heads;
    d.t_q = x.t_q;
    d.causal = x.causal_tail;
    d.seq_lens = x.seq_lens;
    d.max_len = x.max_len;
    d.sm_scale = x.sm_scale;
    d.out = x.out;
    d.lse = x.lse;
    d.k_new = static_cast<const uint16_t *>(x.k16_new);
    d.v_new = static_cast<const uint16_t *>(x.v16_new);
    return prepare_desc(d, x.head_map, need_ptrs, false);
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
                e.layout = sg.layout;
                max_rows = std::max(max_rows, n_new[i] * c->n_kv_heads);
            }
            src += n_new[i];
            ++i;
        }
        if (p.n_entries == 0) continue;
        if (launch_append(p, c->v_type, c->k_type, max_rows, s, pdl) != cudaSuccess) {
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
    const kvq_decode_desc x{c, q16, n_q_heads, t_q, causal_tail, seq_lens, max_len, head_map, sm_scale, out, lse,
                            nullptr, nullptr};
    return kvq_decode_attn_multi(1, &x, workspace, workspace_bytes, stream);
}

kvq_status kvq_decode_workspace_size(const kvq_cache *c, int32_t n_q_heads, int32_t t_q, int32_t max_len,
                                     const int32_t *head_map, size_t *bytes)
{
    const kvq_decode_desc x{c, nullptr, n_q_heads, t_q, 0, nullptr, max_len, head_map, 1.0f, nullptr, nullptr,
                            nullptr, nullptr};
    return kvq_decode_multi_workspace_size(1, &x, bytes);
}

kvq_status kvq_decode_attn_multi(int32_t n, const kvq_decode_desc *calls, void *workspace, size_t workspace_bytes,
                                 void *stream)
{
    if (n < 0 || n > KVQ_MAX_CALLS || (n > 0 && !calls)) return KVQ_ERR_INVALID_ARG;
    std::vector<Desc> ds(n);
    for (int i = 0; i < n; ++i) {
        kvq_status st = to_desc(calls[i], true, ds[i]);
        if (st != KVQ_OK) return st;
        for (int j = 0; j < i; ++j)   // a cache that receives tokens may appear only once
            if (ds[j].c == ds[i].c && (ds[i].k_new || ds[j].k_new)) return KVQ_ERR_INVALID_ARG;
    }
    return run(ds, false, workspace, workspace_bytes, nullptr, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_decode_multi_workspace_size(int32_t n, const kvq_decode_desc *calls, size_t *bytes)
{
    if (!bytes || n < 0 || n > KVQ_MAX_CALLS || (n > 0 && !calls)) return KVQ_ERR_INVALID_ARG;
    std::vector<Desc> ds(n);
    for (int i = 0; i < n; ++i) {
        kvq_status st = to_desc(calls[i], false, ds[i]);
        if (st != KVQ_OK) return st;
    }
    return run(ds, false, nullptr, 0, bytes, nullptr);
}

kvq_status kvq_debug_plan(int32_t n, const kvq_decode_desc *calls, int32_t n_sms, const int32_t *ctas_per_sm,
                          kvq_plan_launch *out, int32_t max_out, int32_t *n_out, size_t *workspace_bytes,
                          int32_t *n_pre_appends)
{
    if (n < 0 || n > KVQ_MAX_CALLS || (n > 0 && !calls) || n_sms < 1 || !ctas_per_sm || max_out < 0 ||
        (max_out > 0 && !out) || !n_out || !workspace_bytes || !n_pre_appends)
        return KVQ_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (ctas_per_sm[i] < 1) return KVQ_ERR_INVALID_ARG;
    std::vector<Desc> ds(n);
    for (int i = 0; i < n; ++i) {
        kvq_status st = to_desc(calls[i], false, ds[i]);
        if (st != KVQ_OK) return st;
        for (int j = 0; j < i; ++j)
            if (ds[j].c == ds[i].c && (ds[i].k_new || ds[j].k_new)) return KVQ_ERR_INVALID_ARG;
    }
    DeviceInfo dev;   // a described device, not a probed one
    dev.n_sms = n_sms;
    for (int kt = 0; kt < 2; ++kt)
        for (int vt = 0; vt < 2; ++vt) {
            dev.ctas[kt][vt][1] = ctas_per_sm[0];
            dev.ctas_half[kt][vt] = ctas_per_sm[1];
            dev.ctas[kt][vt][2] = ctas_per_sm[2];
            dev.ctas[kt][vt][4] = ctas_per_sm[3];
        }
    std::vector<Desc> dsp;
    std::vector<int> pre;
    split_off_pre_appends(ds, dsp, pre);
    std::vector<Launch> lns;
    size_t ws = 0;
    const kvq_status st = plan(dsp, &dev, false, lns, ws);
    if (st != KVQ_OK) return st;
    for (int i = 0; i < (int)lns.size() && i < max_out; ++i) {
        const Launch &ln = lns[i];
        kvq_plan_launch &r = out[i];
        r.kernel = ln.prefill ? 1 : 0;
        r.n_tiles8 = ln.prefill ? 0 : ln.nt;
        r.warps = ln.warps;
        r.chunk = ln.chunk;
        r.chunk0 = ln.chunk0;
        r.n_ctas = ln.n_ctas;
        r.n_rows = ln.n_rows;
    }
    *n_out = (int32_t)lns.size();
    *workspace_bytes = ws;
    *n_pre_appends = (int32_t)pre.size();
    return KVQ_OK;
}

kvq_status kvq_debug_qk(const kvq_cache *c, const void *q16, int32_t n_q_heads, int32_t t_q,
                        const int32_t *seq_lens, int32_t max_len, const int32_t *head_map, int8_t *q_codes,
                        uint16_t *q_scales, int32_t *scores, int32_t *kernel, void *stream)
{
    std::vector<Desc> ds(1);
    Desc &d = ds[0];
    d.c = c;
    d.q = static_cast<const uint16_t *>(q16);
    d.n_q_heads = n_q_heads;
    d.t_q = t_q;
    d.causal = 0;
    d.seq_lens = seq_lens;
    d.max_len = max_len;
    d.sm_scale = 1.0f;
    d.dbg_qc = q_codes;
    d.dbg_qs = q_scales;
    d.dbg_scores = scores;
    kvq_status st = prepare_desc(d, head_map, true, true);
    if (st != KVQ_OK) return st;
    return run(ds, true, nullptr, 0, nullptr, static_cast<cudaStream_t>(stream), kernel);
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

extern "C" kvq_status kvq_debug_lose_stage(const kvq_cache *c, const void *q16, int32_t n_q_heads, int32_t t_q,
                                           int32_t causal_tail, const int32_t *seq_lens, int32_t max_len,
                                           const int32_t *head_map, float sm_scale, float *out, float *lse,
                                           void *workspace, size_t workspace_bytes, void *stream)
{
    const kvq_decode_desc x{c, q16, n_q_heads, t_q, causal_tail, seq_lens, max_len, head_map, sm_scale, out, lse,
                            nullptr, nullptr};
    std::vector<Desc> ds(1);
    const kvq_status st = to_desc(x, true, ds[0]);
    if (st != KVQ_OK) return st;
    return run(ds, false, workspace, workspace_bytes, nullptr, static_cast<cudaStream_t>(stream), nullptr, true);
}

extern "C" kvq_status kvq_reset_wait_timeouts(void)
{
    DeviceInfo *dev = nullptr;
    const kvq_status st = device_setup(&dev);
    if (st != KVQ_OK) return st;
    const unsigned int zero = 0;
    if (cudaMemcpy(dev->timeouts, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

// Coefficients fitted by layout_calib.py on a GB300 (its record
// layout_model.json: 256 kv heads x 60 segments of n tokens, n = 1..32, both
// layouts, least squares of the measured decode times on bytes and unpack
// instructions; the rows permute counted with ncu on the long-context step).
static const kvq_layout_model kDefaultLayoutModel = {8.150755150671073e-08, 2.771975819748976e-06, 134.36};

extern "C" kvq_status kvq_layout_model_default(kvq_layout_model *m)
{
    if (!m) return KVQ_ERR_INVALID_ARG;
    *m = kDefaultLayoutModel;
    return KVQ_OK;
}

extern "C" kvq_status kvq_layout_cost(int32_t layout, int32_t v_type, int32_t n_tokens, const kvq_layout_model *m,
                                      double *cost_us)
{
    if (!cost_us || n_tokens < 1 || (layout != KVQ_LAYOUT_TILES && layout != KVQ_LAYOUT_ROWS) ||
        (v_type != KVQ_V_Q4_0 && v_type != KVQ_V_Q8_0))
        return KVQ_ERR_INVALID_ARG;
    const kvq_layout_model &mm = m ? *m : kDefaultLayoutModel;
    const double code = kD + (v_type == KVQ_V_Q4_0 ? kD / 2 : kD), scales = 2 * kNB * 2;   // bytes per row
    const double tiles = (double)((n_tokens + kWTile - 1) / kWTile);
    double bytes, ops;
    if (layout == KVQ_LAYOUT_TILES) {
        bytes = tiles * kWTile * (code + scales);
        ops = 0.0;
    } else {
        bytes = n_tokens * code + (double)(n_tokens + (n_tokens & 1)) * scales;
        ops = tiles * mm.ops_rows_per_tile;
    }
    *cost_us = mm.us_per_byte * bytes + mm.us_per_op * ops;
    return KVQ_OK;
}

extern "C" kvq_status kvq_choose_layout(int32_t k_type, int32_t v_type, int32_t n_tokens, const kvq_layout_model *m,
                                        int32_t *layout)
{
    if (!layout || (k_type != KVQ_K_I8 && k_type != KVQ_K_F16)) return KVQ_ERR_INVALID_ARG;
    double ct = 0.0, cr = 0.0;
    kvq_status st = kvq_layout_cost(KVQ_LAYOUT_TILES, v_type, n_tokens, m, &ct);
    if (st != KVQ_OK) return st;
    st = kvq_layout_cost(KVQ_LAYOUT_ROWS, v_type, n_tokens, m, &cr);
    if (st != KVQ_OK) return st;
    *layout = (k_type == KVQ_K_I8 && cr < ct) ? KVQ_LAYOUT_ROWS : KVQ_LAYOUT_TILES;
    return KVQ_OK;
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
