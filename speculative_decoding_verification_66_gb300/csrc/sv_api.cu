// sv_api.cu -- the C ABI (include/spec_verify.h): argument checks, launch
// planning, workspace carving and the three launches.
#include <cmath>
#include <cstring>
#include <mutex>

#include "spec_verify.h"
#include "sv_internal.h"

#define SV_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

using sv::Geometry;

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;

size_t round_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct DeviceCache {
    bool ready = false;
    int sms = 0;
    int blocks[2][2] = {{0, 0}, {0, 0}};  // pass-1 CTAs per SM, [es == 2][mode]
    int sample_blocks[2] = {0, 0};        // sampler CTAs per SM, [es == 2]
    int filter_blocks[2] = {0, 0};        // filter CTAs per SM, [es == 2]
};
std::mutex g_mu;
DeviceCache g_cache[kMaxDevices];

// SM count, resident pass-1 CTAs per SM and resident sampler CTAs per SM on
// the current device.
int device_limits(int es, int mode, int* sms, int* blocks, int* sample_blocks)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceCache& c = g_cache[dev];
    if (!c.ready) {
        if (cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SV_ERR_CUDA;
        for (int e = 0; e < 2; ++e)
            for (int m = 0; m < 2; ++m)
                if (sv::row_stats_blocks_per_sm(e ? 2 : 4, m, &c.blocks[e][m]) != cudaSuccess)
                    return SV_ERR_CUDA;
        for (int e = 0; e < 2; ++e)
            if (sv::sample_blocks_per_sm(e ? 2 : 4, &c.sample_blocks[e]) != cudaSuccess)
                return SV_ERR_CUDA;
        for (int e = 0; e < 2; ++e)
            if (sv::filter_blocks_per_sm(e ? 2 : 4, &c.filter_blocks[e]) != cudaSuccess)
                return SV_ERR_CUDA;
        c.ready = true;
    }
    *sms = c.sms;
    *blocks = c.blocks[es == 2][mode];
    *sample_blocks = c.sample_blocks[es == 2];
    return (*sms > 0 && *blocks > 0 && *sample_blocks > 0 && c.filter_blocks[es == 2] > 0)
               ? SV_OK
               : SV_ERR_CUDA;
}

// Resident filter CTAs per SM on the current device (after device_limits).
int filter_blocks(int es)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    return g_cache[dev].ready ? g_cache[dev].sms * g_cache[dev].filter_blocks[es == 2] : 0;
}

struct Layout {
    size_t partials = 0, seqs = 0, block_sums = 0, total = 0;
    // Early exit only.
    size_t still = 0, lists = 0, counters = 0, counter_bytes = 0;
    // Sharded only.
    size_t pairs = 0;
    // Filtered only: one FiltRow per row.
    size_t filt = 0;
};

// Early exit: the positions 0 .. K are verified in phases of 1, 2, 4, ...
// positions; phase k covers target rows [p0, p0 + nt) and draft rows
// [p0, p0 + nd) of the sequences still undecided after phase k - 1.
struct Phase {
    int32_t p0, nt, nd;
};
constexpr int kMaxPhases = 16;  // K <= 1024 needs at most 11

int plan_phases(int64_t K, bool sampling, Phase* ph)
{
    int n = 0;
    int64_t p0 = 0, len = 1;
    while (p0 <= K) {
        const int64_t nt = len < K + 1 - p0 ? len : K + 1 - p0;
        int64_t nd = 0;
        if (sampling) nd = len < K - p0 ? len : (K - p0 > 0 ? K - p0 : 0);
        ph[n++] = Phase{static_cast<int32_t>(p0), static_cast<int32_t>(nt), static_cast<int32_t>(nd)};
        p0 += len;
        len *= 2;
    }
    return n;
}

int check_sizes(int64_t B, int64_t K, int64_t V, int dtype, int mode)
{
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_DTYPE;
    if (mode != SV_SAMPLE && mode != SV_GREEDY) return SV_ERR_ARG;
    if (B < 0 || K < 0 || V < 1) return SV_ERR_ARG;
    if (B >= (int64_t(1) << 31) || K > sv::kMaxK || V >= (int64_t(1) << 31)) return SV_ERR_SIZE;
    const int64_t es = dtype == SV_BF16 ? 2 : 4;
    // B (2K + 1) V es < 2^62, checked without overflow.
    const int64_t per_seq = (2 * K + 1) * V * es;  // < 2^11 * 2^31 * 4 = 2^44
    if (B > 0 && per_seq > (int64_t(1) << 62) / B) return SV_ERR_SIZE;
    return SV_OK;
}

int make_plan(int64_t B, int64_t K, int64_t V, int dtype, int mode, Geometry* g, Layout* L,
              bool early_exit = false, int shards = 1, bool filtered = false)
{
    int rc = check_sizes(B, K, V, dtype, mode);
    if (rc != SV_OK) return rc;
    const int es = dtype == SV_BF16 ? 2 : 4;
    int sms = 0, blocks = 0, sample_blocks = 0;
    rc = device_limits(es, mode, &sms, &blocks, &sample_blocks);
    if (rc != SV_OK) return rc;

    std::memset(g, 0, sizeof(*g));
    g->B = B;
    g->K = K;
    g->V = V;
    g->es = es;
    g->mode = mode;
    g->rows_t = B * (K + 1);
    g->rows = g->rows_t + (mode == SV_SAMPLE ? B * K : 0);
    g->aligned = (V * es) % 16 == 0;
    // Pass 1 streams logical rows (shard copies split at the boundaries), or
    // each shard row when shard rows are not 16-byte aligned.
    g->shards = shards;
    g->shard_len = V / shards;
    g->shard_aligned = (g->shard_len * es) % 16 == 0;
    g->row_shards = (g->shard_aligned && g->shard_len * es >= 4096) ? 1 : shards;
    g->row_len = g->row_shards == 1 ? V : g->shard_len;
    g->row_aligned = (g->row_len * es) % 16 == 0;
    // Misaligned rows need one extra 16-byte vector per tile in the buffer.
    g->tile_elems = (g->row_aligned ? sv::kRowTileBytes : sv::kRowTileBytes - 16) / es;
    g->tiles_per_row = (g->row_len + g->tile_elems - 1) / g->tile_elems;
    g->tiles = g->rows * g->row_shards * g->tiles_per_row;
    if (early_exit) {
        // The grid and the partials serve every phase: size them for the
        // phase with the most rows per sequence, as if all B took part.
        Phase ph[kMaxPhases];
        const int nph = plan_phases(K, mode == SV_SAMPLE, ph);
        int64_t most = 0;
        for (int k = 0; k < nph; ++k)
            most = ph[k].nt + ph[k].nd > most ? ph[k].nt + ph[k].nd : most;
        g->tiles = B * most * g->row_shards * g->tiles_per_row;
    }
    const int64_t want = static_cast<int64_t>(sms) * blocks;
    g->grid = static_cast<int32_t>(g->tiles < want ? (g->tiles > 0 ? g->tiles : 1) : want);
    const int64_t per_cta = (g->tiles + g->grid - 1) / g->grid;
    g->maxseg = static_cast<int32_t>((per_cta + g->tiles_per_row - 1) / g->tiles_per_row + 1);
    g->nblocks = (V + sv::kRaceBlock - 1) / sv::kRaceBlock;
    const int64_t tok = sv::sample_tokens_per_slice(es);
    const int64_t slices = B * ((V + tok - 1) / tok);  // < 2^62 / 2048: no overflow
    const int64_t warps_per_cta = sv::kSampleThreads / 32;
    const int64_t want_s = static_cast<int64_t>(sms) * sample_blocks;
    const int64_t need_s = (slices + warps_per_cta - 1) / warps_per_cta;
    g->sample_grid = static_cast<int32_t>(need_s < want_s ? (need_s > 0 ? need_s : 1) : want_s);

    size_t off = 0;
    L->partials = off;
    off += round_up(static_cast<size_t>(g->grid) * g->maxseg * sv::kRowConsumerWarps *
                    sizeof(sv::Partial));
    L->seqs = off;
    off += round_up(static_cast<size_t>(B) * sizeof(sv::SeqRecord));
    L->block_sums = off;
    if (mode == SV_SAMPLE) off += round_up(static_cast<size_t>(B * g->nblocks) * sizeof(float));
    if (shards > 1 && mode == SV_SAMPLE && !g->shard_aligned) {
        // The emitted row pairs gathered from the shards, [B][2][V] (shard
        // widths that are not whole 16-byte vectors only).
        L->pairs = off;
        off += round_up(static_cast<size_t>(2 * B) * static_cast<size_t>(V) * es);
    }
    if (filtered && mode == SV_SAMPLE) {
        L->filt = off;
        off += round_up(static_cast<size_t>(g->rows) * sizeof(sv::FiltRow));
    }
    if (early_exit) {
        L->still = off;
        off += round_up(static_cast<size_t>(B) * sizeof(int32_t));
        L->lists = off;
        off += round_up(2 * static_cast<size_t>(B) * sizeof(int32_t));
        L->counters = off;  // per phase: the next count, then the ticket
        L->counter_bytes = 2 * kMaxPhases * sizeof(int32_t);
        off += round_up(L->counter_bytes);
    }
    L->total = off > 0 ? off : kAlign;
    return SV_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int run(const void* target, const void* draft, const int32_t* tokens, int64_t B, int64_t K,
        int64_t V, int dtype, float temperature, uint64_t seed, int mode, int32_t* out_tokens,
        int32_t* num_accepted, void* workspace, size_t workspace_bytes, void* stream,
        double* lse_t, double* lse_d, double* log_ratio, int32_t* seq_status,
        void* const* events, int n_events, bool early_exit = false,
        const void* const* t_shards = nullptr, const void* const* d_shards = nullptr, int G = 1,
        int64_t top_k = 0, float top_p = 1.0f, float* thr_t = nullptr, float* thr_d = nullptr)
{
    int rc = check_sizes(B, K, V, dtype, mode);
    if (rc != SV_OK) return rc;
    if (top_k < 0 || !(top_p > 0.f && top_p <= 1.f)) return SV_ERR_ARG;
    // Filtering changes sampling only (the cuts keep every row's maximum).
    const bool filtered = mode == SV_SAMPLE && ((top_k > 0 && top_k < V) || top_p < 1.f);
    float c = 0.f;
    if (mode == SV_SAMPLE) {
        if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_ARG;
        c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
        if (!std::isfinite(c) || !(c > 0.f)) return SV_ERR_ARG;
    }
    if (events != nullptr && n_events < 4) return SV_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto record = [&](int i) -> bool {
        return events == nullptr ||
               cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    };
    if (B == 0) {
        for (int i = 0; i < 4; ++i)
            if (!record(i)) return SV_ERR_CUDA;
        return SV_OK;
    }
    const bool sampling = mode == SV_SAMPLE;
    if (t_shards != nullptr || G > 1) {
        // Sharded: every shard must be given and 16-byte aligned; shard 0
        // stands for the tensors in the checks below.
        if (G < 1 || G > sv::kMaxShards || t_shards == nullptr ||
            (sampling && K > 0 && d_shards == nullptr))
            return SV_ERR_ARG;
        for (int gi = 0; gi < G; ++gi) {
            if (t_shards[gi] == nullptr || (sampling && K > 0 && d_shards[gi] == nullptr))
                return SV_ERR_ARG;
            if (!aligned_to(t_shards[gi], 16) || (sampling && K > 0 && !aligned_to(d_shards[gi], 16)))
                return SV_ERR_ALIGN;
        }
        target = t_shards[0];
        draft = sampling && K > 0 ? d_shards[0] : nullptr;
    }
    if (target == nullptr || out_tokens == nullptr || num_accepted == nullptr) return SV_ERR_ARG;
    if (K > 0 && tokens == nullptr) return SV_ERR_ARG;
    if (sampling && K > 0 && draft == nullptr) return SV_ERR_ARG;
    if (workspace == nullptr) return SV_ERR_WORKSPACE;
    if (!aligned_to(target, 16) || (sampling && K > 0 && !aligned_to(draft, 16))) return SV_ERR_ALIGN;
    if ((tokens && !aligned_to(tokens, 4)) || !aligned_to(out_tokens, 4) ||
        !aligned_to(num_accepted, 4) || (seq_status && !aligned_to(seq_status, 4)))
        return SV_ERR_ALIGN;
    if ((lse_t && !aligned_to(lse_t, 8)) || (lse_d && !aligned_to(lse_d, 8)) ||
        (log_ratio && !aligned_to(log_ratio, 8)) || (thr_t && !aligned_to(thr_t, 4)) ||
        (thr_d && !aligned_to(thr_d, 4)))
        return SV_ERR_ALIGN;
    if (!aligned_to(workspace, kAlign)) return SV_ERR_WORKSPACE;

    Geometry g;
    Layout L;
    rc = make_plan(B, K, V, dtype, mode, &g, &L, early_exit, G, filtered);
    if (rc != SV_OK) return rc;
    if (workspace_bytes < L.total) return SV_ERR_WORKSPACE;
    if (filtered && (early_exit || G > 1)) return SV_ERR_ARG;
    // Events between the kernels would sit between programmatically chained
    // launches; the timed variant launches them one after the other instead.
    g.pdl = events == nullptr ? 1 : 0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    const uint8_t* tp = static_cast<const uint8_t*>(target);
    const uint8_t* dp = sampling ? static_cast<const uint8_t*>(draft) : nullptr;
    auto* partials = reinterpret_cast<sv::Partial*>(ws + L.partials);
    auto* seqs = reinterpret_cast<sv::SeqRecord*>(ws + L.seqs);
    auto* block_sums = reinterpret_cast<float*>(ws + L.block_sums);

    const sv::RowMap full{nullptr, nullptr, 0, static_cast<int32_t>(K + 1),
                          static_cast<int32_t>(sampling ? K : 0)};
    sv::Shards sh{};
    for (int gi = 0; gi < G; ++gi) {
        sh.t[gi] = static_cast<const uint8_t*>(t_shards != nullptr ? t_shards[gi] : target);
        sh.d[gi] = dp == nullptr ? nullptr
                                 : static_cast<const uint8_t*>(d_shards != nullptr ? d_shards[gi] : draft);
    }
    const int64_t row_bytes = V * g.es;
    sv::RowPairLayout lay{K + 1, 1, K, 1, tp + g.rows_t * row_bytes,
                          dp != nullptr ? dp + B * K * row_bytes : nullptr};
    const uint8_t* sp_t = tp;
    const uint8_t* sp_d = dp;
    const bool direct = G > 1 && g.shard_aligned;
    if (G > 1 && sampling && !direct) {
        // The sampler reads the emitted pairs gathered from the shards.
        uint8_t* pairs = ws + L.pairs;
        sp_t = pairs;
        sp_d = pairs + row_bytes;
        lay = sv::RowPairLayout{2, 0, 2, 0, pairs + 2 * B * row_bytes, pairs + 2 * B * row_bytes};
    }
    sv::RowStatsArgs ra{tp, dp, g, c, partials, full, sh};
    sv::ScanArgs sa{tp, dp, tokens, g, c, seed, partials, out_tokens, num_accepted, seqs,
                    sampling ? lse_t : nullptr, sampling ? lse_d : nullptr,
                    sampling ? log_ratio : nullptr, seq_status, full, nullptr,
                    sampling ? thr_t : nullptr, sampling ? thr_d : nullptr,
                    nullptr, nullptr, nullptr, nullptr, sh};
    sv::SampleArgs pa{sp_t, sp_d, g, c, seed, seqs, block_sums,
                      out_tokens, num_accepted, seq_status, lay, direct ? 1 : 0, sh, 0};
    sv::GatherArgs ga{g, sh, seqs, ws + L.pairs};

    if (filtered) {
        // Thresholds and kept-mass normalisers of every row replace pass 1.
        auto* filt = reinterpret_cast<sv::FiltRow*>(ws + L.filt);
        const int64_t cap = filter_blocks(g.es);
        if (cap <= 0) return SV_ERR_CUDA;
        const int grid = static_cast<int>(g.rows < cap ? g.rows : cap);
        sv::FilterArgs fa{tp, dp, g, c, top_k, top_p, filt};
        sa.filt = filt;
        pa.filtered = 1;
        if (!record(0)) return SV_ERR_CUDA;
        if (sv::launch_filter(fa, grid, s) != cudaSuccess) return SV_ERR_CUDA;
        if (!record(1)) return SV_ERR_CUDA;
        if (sv::launch_scan(sa, s) != cudaSuccess) return SV_ERR_CUDA;
        if (!record(2)) return SV_ERR_CUDA;
        if (sv::launch_sample(pa, s) != cudaSuccess) return SV_ERR_CUDA;
        if (!record(3)) return SV_ERR_CUDA;
        return SV_OK;
    }

    if (early_exit) {
        // Phases over the positions; each pass 1 reads only the rows of the
        // sequences the previous scan left undecided.
        auto* still = reinterpret_cast<int32_t*>(ws + L.still);
        auto* lists = reinterpret_cast<int32_t*>(ws + L.lists);
        auto* counters = reinterpret_cast<int32_t*>(ws + L.counters);
        if (cudaMemsetAsync(counters, 0, L.counter_bytes, s) != cudaSuccess) return SV_ERR_CUDA;
        Phase ph[kMaxPhases];
        const int nph = plan_phases(K, sampling, ph);
        for (int k = 0; k < nph; ++k) {
            sv::RowMap mp{nullptr, nullptr, ph[k].p0, ph[k].nt, ph[k].nd};
            if (k > 0) {
                mp.active = lists + ((k - 1) & 1) * B;
                mp.count = counters + (k - 1);
            }
            ra.map = mp;
            sa.map = mp;
            const bool last = k == nph - 1;
            sa.still = last ? nullptr : still;
            sa.next_active = last ? nullptr : lists + (k & 1) * B;
            sa.next_count = last ? nullptr : counters + k;
            sa.ticket = last ? nullptr : reinterpret_cast<uint32_t*>(counters + kMaxPhases + k);
            if (sv::launch_row_stats(ra, s) != cudaSuccess) return SV_ERR_CUDA;
            if (sv::launch_scan(sa, s) != cudaSuccess) return SV_ERR_CUDA;
        }
        if (sampling && sv::launch_sample(pa, s) != cudaSuccess) return SV_ERR_CUDA;
        return SV_OK;
    }

    if (!record(0)) return SV_ERR_CUDA;
    if (sv::launch_row_stats(ra, s) != cudaSuccess) return SV_ERR_CUDA;
    if (!record(1)) return SV_ERR_CUDA;
    if (sv::launch_scan(sa, s) != cudaSuccess) return SV_ERR_CUDA;
    if (!record(2)) return SV_ERR_CUDA;
    if (sampling && G > 1 && !direct && sv::launch_gather_pairs(ga, s) != cudaSuccess)
        return SV_ERR_CUDA;
    if (sampling && sv::launch_sample(pa, s) != cudaSuccess) return SV_ERR_CUDA;
    if (!record(3)) return SV_ERR_CUDA;
    return SV_OK;
}

struct HostLayout {
    size_t target = 0, draft = 0, tokens = 0, out = 0, nacc = 0, ws = 0, total = 0;
    size_t target_bytes = 0, draft_bytes = 0, tokens_bytes = 0, out_bytes = 0, nacc_bytes = 0;
    size_t ws_bytes = 0;
};

int host_layout(int64_t B, int64_t K, int64_t V, int dtype, int mode, HostLayout* h)
{
    int rc = check_sizes(B, K, V, dtype, mode);
    if (rc != SV_OK) return rc;
    Geometry g;
    Layout L;
    rc = make_plan(B, K, V, dtype, mode, &g, &L);
    if (rc != SV_OK) return rc;
    const size_t es = dtype == SV_BF16 ? 2 : 4;
    h->target_bytes = static_cast<size_t>(B * (K + 1) * V) * es;
    h->draft_bytes = mode == SV_SAMPLE ? static_cast<size_t>(B * K * V) * es : 0;
    h->tokens_bytes = static_cast<size_t>(B * K) * 4;
    h->out_bytes = static_cast<size_t>(B * (K + 1)) * 4;
    h->nacc_bytes = static_cast<size_t>(B) * 4;
    h->ws_bytes = L.total;
    size_t off = 0;
    h->target = off;
    off += round_up(h->target_bytes);
    h->draft = off;
    off += round_up(h->draft_bytes);
    h->tokens = off;
    off += round_up(h->tokens_bytes);
    h->out = off;
    off += round_up(h->out_bytes);
    h->nacc = off;
    off += round_up(h->nacc_bytes);
    h->ws = off;
    off += round_up(h->ws_bytes);
    h->total = off;
    return SV_OK;
}

}  // namespace

SV_EXPORT int sv_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode, size_t* bytes)
{
    if (bytes == nullptr) return SV_ERR_ARG;
    Geometry g;
    Layout L;
    const int rc = make_plan(B, K, V, dtype, mode, &g, &L);
    if (rc != SV_OK) return rc;
    *bytes = L.total;
    return SV_OK;
}

SV_EXPORT int spec_verify(const void* target_logits, const void* draft_logits,
                          const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V, int dtype,
                          float temperature, uint64_t seed, int mode, int32_t* out_tokens,
                          int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                          void* stream)
{
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, nullptr, nullptr, 0);
}

SV_EXPORT int sv_early_exit_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode,
                                            size_t* bytes)
{
    if (bytes == nullptr) return SV_ERR_ARG;
    Geometry g;
    Layout L;
    const int rc = make_plan(B, K, V, dtype, mode, &g, &L, true);
    if (rc != SV_OK) return rc;
    *bytes = L.total;
    return SV_OK;
}

SV_EXPORT int spec_verify_early_exit(const void* target_logits, const void* draft_logits,
                                     const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                     int dtype, float temperature, uint64_t seed, int mode,
                                     int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                     size_t workspace_bytes, void* stream)
{
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, nullptr, nullptr, 0, true);
}

SV_EXPORT int sv_sharded_workspace_bytes(int64_t B, int64_t K, int64_t Vs, int G, int dtype, int mode,
                                         size_t* bytes)
{
    if (bytes == nullptr || G < 1 || G > sv::kMaxShards || Vs < 1) return SV_ERR_ARG;
    if (Vs >= (int64_t(1) << 31)) return SV_ERR_SIZE;
    Geometry g;
    Layout L;
    const int rc = make_plan(B, K, G * Vs, dtype, mode, &g, &L, false, G);
    if (rc != SV_OK) return rc;
    *bytes = L.total;
    return SV_OK;
}

SV_EXPORT int spec_verify_sharded(const void* const* target_shards, const void* const* draft_shards,
                                  int G, const int32_t* draft_tokens, int64_t B, int64_t K,
                                  int64_t Vs, int dtype, float temperature, uint64_t seed, int mode,
                                  int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                  size_t workspace_bytes, void* stream)
{
    if (G < 1 || G > sv::kMaxShards || Vs < 1) return SV_ERR_ARG;
    if (Vs >= (int64_t(1) << 31)) return SV_ERR_SIZE;
    const int64_t V = G * Vs;
    // The pair gather puts 256 vectors per CTA on grid y (at most 65535).
    const int64_t per_chunk = 256 * (dtype == SV_BF16 ? 8 : 4);
    if (G > 1 && (V + per_chunk - 1) / per_chunk > 65535) return SV_ERR_SIZE;
    if (B > 0 && target_shards == nullptr) return SV_ERR_ARG;
    return run(nullptr, nullptr, draft_tokens, B, K, V, dtype, temperature, seed, mode, out_tokens,
               num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr,
               nullptr, 0, false, target_shards, draft_shards, G);
}

SV_EXPORT int sv_filtered_workspace_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode,
                                         size_t* bytes)
{
    if (bytes == nullptr) return SV_ERR_ARG;
    Geometry g;
    Layout L;
    const int rc = make_plan(B, K, V, dtype, mode, &g, &L, false, 1, true);
    if (rc != SV_OK) return rc;
    *bytes = L.total;
    return SV_OK;
}

SV_EXPORT int spec_verify_filtered(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                   int dtype, float temperature, int64_t top_k, float top_p,
                                   uint64_t seed, int mode, int32_t* out_tokens,
                                   int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                                   void* stream)
{
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, nullptr, nullptr, 0, false, nullptr, nullptr, 1, top_k, top_p);
}

SV_EXPORT int spec_verify_filtered_debug(const void* target_logits, const void* draft_logits,
                                         const int32_t* draft_tokens, int64_t B, int64_t K,
                                         int64_t V, int dtype, float temperature, int64_t top_k,
                                         float top_p, uint64_t seed, int mode,
                                         int32_t* out_tokens, int32_t* num_accepted,
                                         void* workspace, size_t workspace_bytes, void* stream,
                                         double* lse_t, double* lse_d, float* thr_t, float* thr_d,
                                         int32_t* seq_status)
{
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, lse_t, lse_d, nullptr,
               seq_status, nullptr, 0, false, nullptr, nullptr, 1, top_k, top_p, thr_t, thr_d);
}

SV_EXPORT int spec_verify_filtered_timed(const void* target_logits, const void* draft_logits,
                                         const int32_t* draft_tokens, int64_t B, int64_t K,
                                         int64_t V, int dtype, float temperature, int64_t top_k,
                                         float top_p, uint64_t seed, int mode,
                                         int32_t* out_tokens, int32_t* num_accepted,
                                         void* workspace, size_t workspace_bytes, void* stream,
                                         void* const* events, int n_events)
{
    if (events == nullptr) return SV_ERR_ARG;
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, nullptr, events, n_events, false, nullptr, nullptr, 1, top_k, top_p);
}

SV_EXPORT int spec_verify_debug(const void* target_logits, const void* draft_logits,
                                const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                int dtype, float temperature, uint64_t seed, int mode,
                                int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                size_t workspace_bytes, void* stream, double* lse_t, double* lse_d,
                                double* log_ratio, int32_t* seq_status)
{
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, lse_t, lse_d,
               log_ratio, seq_status, nullptr, 0);
}

SV_EXPORT int spec_verify_timed(const void* target_logits, const void* draft_logits,
                                const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                int dtype, float temperature, uint64_t seed, int mode,
                                int32_t* out_tokens, int32_t* num_accepted, void* workspace,
                                size_t workspace_bytes, void* stream, void* const* events,
                                int n_events)
{
    if (events == nullptr) return SV_ERR_ARG;
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, nullptr, events, n_events);
}

SV_EXPORT int sv_host_staging_bytes(int64_t B, int64_t K, int64_t V, int dtype, int mode,
                                    size_t* bytes)
{
    if (bytes == nullptr) return SV_ERR_ARG;
    HostLayout h;
    const int rc = host_layout(B, K, V, dtype, mode, &h);
    if (rc != SV_OK) return rc;
    *bytes = h.total;
    return SV_OK;
}

SV_EXPORT int spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                               const int32_t* h_draft_tokens, int64_t B, int64_t K, int64_t V,
                               int dtype, float temperature, uint64_t seed, int mode,
                               int32_t* h_out_tokens, int32_t* h_num_accepted, void* staging,
                               size_t staging_bytes, void* stream)
{
    HostLayout h;
    int rc = host_layout(B, K, V, dtype, mode, &h);
    if (rc != SV_OK) return rc;
    if (B == 0) return SV_OK;
    const bool sampling = mode == SV_SAMPLE;
    if (h_target_logits == nullptr || h_out_tokens == nullptr || h_num_accepted == nullptr)
        return SV_ERR_ARG;
    if (K > 0 && h_draft_tokens == nullptr) return SV_ERR_ARG;
    if (sampling && K > 0 && h_draft_logits == nullptr) return SV_ERR_ARG;
    if (staging == nullptr || !aligned_to(staging, kAlign) || staging_bytes < h.total)
        return SV_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* st = static_cast<uint8_t*>(staging);
    if (cudaMemcpyAsync(st + h.target, h_target_logits, h.target_bytes, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return SV_ERR_CUDA;
    if (h.draft_bytes > 0 &&
        cudaMemcpyAsync(st + h.draft, h_draft_logits, h.draft_bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
        return SV_ERR_CUDA;
    if (h.tokens_bytes > 0 &&
        cudaMemcpyAsync(st + h.tokens, h_draft_tokens, h.tokens_bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
        return SV_ERR_CUDA;
    rc = spec_verify(st + h.target, sampling ? st + h.draft : nullptr,
                     reinterpret_cast<const int32_t*>(st + h.tokens), B, K, V, dtype, temperature,
                     seed, mode, reinterpret_cast<int32_t*>(st + h.out),
                     reinterpret_cast<int32_t*>(st + h.nacc), st + h.ws, h.ws_bytes, stream);
    if (rc != SV_OK) return rc;
    if (cudaMemcpyAsync(h_out_tokens, st + h.out, h.out_bytes, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(h_num_accepted, st + h.nacc, h.nacc_bytes, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

SV_EXPORT const char* sv_error_string(int code)
{
    switch (code) {
        case SV_OK: return "success";
        case SV_ERR_ARG: return "invalid argument (size, mode, temperature or NULL pointer)";
        case SV_ERR_DTYPE: return "unknown logits dtype";
        case SV_ERR_ALIGN: return "misaligned pointer (logits need 16 bytes, int32 buffers 4)";
        case SV_ERR_WORKSPACE: return "workspace or staging buffer NULL, too small or not 256-byte aligned";
        case SV_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case SV_ERR_SIZE: return "sizes outside the supported range";
        default: return "unknown status code";
    }
}

SV_EXPORT int sv_version(void) { return 104; }
