// sv_api.cu -- the C ABI (include/spec_verify.h): argument checks, launch
// planning, workspace carving and the three launches.
#include <cmath>
#include <cstring>
#include <mutex>

#include "spec_verify.h"
#include "sv_stages.h"

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
    // Shard rows that fit a tile are a tile each: one bulk copy per tile
    // instead of two pieces from two shards.
    if (shards > 1 && g->row_shards == 1 && g->shard_len * es <= sv::kRowTileBytes)
        g->tile_elems = g->shard_len;
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
        int64_t top_k = 0, float top_p = 1.0f, float* thr_t = nullptr, float* thr_d = nullptr,
        const int32_t* gate = nullptr, int gate_stage = 0)
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
    // The thresholds kernels' fixed-point mass sums (2^40 per token at most)
    // hold rows below 2^22 tokens.
    if (filtered && V >= (int64_t(1) << 22)) return SV_ERR_SIZE;
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
    // Test hook: stage 1 holds pass 1's (or the thresholds kernel's) copies,
    // stage 2 the sampler's.
    sv::RowStatsArgs ra{tp, dp, g, c, partials, full, sh, gate_stage == 1 ? gate : nullptr};
    sv::ScanArgs sa{tp, dp, tokens, g, c, seed, partials, out_tokens, num_accepted, seqs,
                    sampling ? lse_t : nullptr, sampling ? lse_d : nullptr,
                    sampling ? log_ratio : nullptr, seq_status, full, nullptr,
                    sampling ? thr_t : nullptr, sampling ? thr_d : nullptr,
                    nullptr, nullptr, nullptr, nullptr, sh};
    sv::SampleArgs pa{sp_t, sp_d, g, c, seed, seqs, block_sums,
                      out_tokens, num_accepted, seq_status, lay, direct ? 1 : 0, sh, 0,
                      gate_stage == 2 ? gate : nullptr};
    sv::GatherArgs ga{g, sh, seqs, ws + L.pairs};

    if (filtered) {
        // Thresholds and kept-mass normalisers of every row replace pass 1.
        auto* filt = reinterpret_cast<sv::FiltRow*>(ws + L.filt);
        const int64_t cap = filter_blocks(g.es);
        if (cap <= 0) return SV_ERR_CUDA;
        const int grid = static_cast<int>(g.rows < cap ? g.rows : cap);
        int sms = 0, blocks = 0, sample_blocks = 0;
        if (device_limits(g.es, mode, &sms, &blocks, &sample_blocks) != SV_OK) return SV_ERR_CUDA;
        sv::FilterArgs fa{tp, dp, g, c, top_k, top_p, filt, gate_stage == 1 ? gate : nullptr};
        sa.filt = filt;
        pa.filtered = 1;
        if (!record(0)) return SV_ERR_CUDA;
        if (sv::launch_filter(fa, grid, sms, s) != cudaSuccess) return SV_ERR_CUDA;
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

SV_EXPORT int spec_verify_gated(const void* target_logits, const void* draft_logits,
                                const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                int dtype, float temperature, int64_t top_k, float top_p,
                                uint64_t seed, int mode, int32_t* out_tokens,
                                int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                                void* stream, int32_t* seq_status, int stage, const int32_t* gate)
{
    if (gate == nullptr || (stage != 1 && stage != 2)) return SV_ERR_ARG;
    if (!aligned_to(gate, 4)) return SV_ERR_ALIGN;
    return run(target_logits, draft_logits, draft_tokens, B, K, V, dtype, temperature, seed, mode,
               out_tokens, num_accepted, workspace, workspace_bytes, stream, nullptr, nullptr,
               nullptr, seq_status, nullptr, 0, false, nullptr, nullptr, 1, top_k, top_p, nullptr,
               nullptr, gate, stage);
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

// ---------------------------------------------------------------------------
// LM head fused with the row statistics.
// ---------------------------------------------------------------------------
namespace {

struct LmLayout {
    size_t part = 0, tok = 0, seqs = 0, block_sums = 0, err = 0, ht = 0, hd = 0, pairs = 0;
    size_t total = 0;
    int64_t rows = 0, n_vt = 0;
};

int lm_check_sizes(int64_t B, int64_t K, int64_t V, int64_t Dt, int64_t Dd, int mode)
{
    int rc = check_sizes(B, K, V, SV_F32, mode);
    if (rc != SV_OK) return rc;
    const bool draft = mode == SV_SAMPLE && K > 0;
    if (Dt < 8 || Dt % 8 != 0 || (draft && (Dd < 8 || Dd % 8 != 0))) return SV_ERR_ARG;
    // Tensor-map limits: extents below 2^32, row strides (2 D bytes) below 2^40.
    if (Dt >= (int64_t(1) << 31) || Dd >= (int64_t(1) << 31)) return SV_ERR_SIZE;
    if (B * (K + 1) >= (int64_t(1) << 31)) return SV_ERR_SIZE;
    return SV_OK;
}

int lm_plan(int64_t B, int64_t K, int64_t V, int64_t Dt, int64_t Dd, int mode, Geometry* g,
            LmLayout* L)
{
    int rc = lm_check_sizes(B, K, V, Dt, Dd, mode);
    if (rc != SV_OK) return rc;
    Layout base;
    rc = make_plan(B, K, V, SV_F32, mode, g, &base);
    if (rc != SV_OK) return rc;
    const bool sampling = mode == SV_SAMPLE;
    L->n_vt = sv::lmhead_vocab_tiles(V);
    L->rows = B * (K + 1) + (sampling ? B * K : 0);
    size_t off = 0;
    L->part = off;
    off += round_up(static_cast<size_t>(L->rows) * static_cast<size_t>(L->n_vt) * sizeof(sv::Partial));
    L->tok = off;
    off += round_up(static_cast<size_t>(L->rows) * sizeof(float));
    L->seqs = off;
    off += round_up(static_cast<size_t>(B) * sizeof(sv::SeqRecord));
    L->err = off;
    off += round_up(sizeof(int32_t));
    if (sampling) {
        L->block_sums = off;
        off += round_up(static_cast<size_t>(B * g->nblocks) * sizeof(float));
        L->ht = off;
        off += round_up(static_cast<size_t>(B * Dt) * 2);
        L->hd = off;
        off += round_up(static_cast<size_t>(B * (K > 0 ? Dd : 8)) * 2);
        L->pairs = off;
        off += round_up(static_cast<size_t>(2 * B) * static_cast<size_t>(V) * sizeof(float));
    }
    L->total = off;
    return SV_OK;
}

// Stats GEMM -> scan -> (sampling) emitted hidden states -> logits of the
// emitted row pairs -> sampler; the LM head's timeout check last. Events
// (5): before the stats GEMM, after it, after the scan, after the emitted
// pairs' GEMM, at the end.
int run_lmhead(const void* hidden_t, const void* w_t, const void* hidden_d, const void* w_d,
               const int32_t* tokens, int64_t B, int64_t K, int64_t V, int64_t Dt, int64_t Dd,
               float temperature, uint64_t seed, int mode, int32_t* out_tokens,
               int32_t* num_accepted, void* workspace, size_t workspace_bytes, void* stream,
               double* lse_t, double* lse_d, double* log_ratio, int32_t* seq_status,
               void* const* events, int n_events, const int32_t* gate = nullptr)
{
    int rc = lm_check_sizes(B, K, V, Dt, Dd, mode);
    if (rc != SV_OK) return rc;
    const bool sampling = mode == SV_SAMPLE;
    float c = 0.f;
    if (sampling) {
        if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_ARG;
        c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
        if (!std::isfinite(c) || !(c > 0.f)) return SV_ERR_ARG;
    }
    if (events != nullptr && n_events < 5) return SV_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto record = [&](int i) -> bool {
        return events == nullptr ||
               cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    };
    if (B == 0) {
        for (int i = 0; i < 5; ++i)
            if (!record(i)) return SV_ERR_CUDA;
        return SV_OK;
    }
    const bool with_draft = sampling && K > 0;
    if (hidden_t == nullptr || w_t == nullptr || out_tokens == nullptr || num_accepted == nullptr)
        return SV_ERR_ARG;
    if (K > 0 && tokens == nullptr) return SV_ERR_ARG;
    if (with_draft && (hidden_d == nullptr || w_d == nullptr)) return SV_ERR_ARG;
    if (workspace == nullptr) return SV_ERR_WORKSPACE;
    if (!aligned_to(hidden_t, 16) || !aligned_to(w_t, 16) ||
        (with_draft && (!aligned_to(hidden_d, 16) || !aligned_to(w_d, 16))))
        return SV_ERR_ALIGN;
    if ((tokens && !aligned_to(tokens, 4)) || !aligned_to(out_tokens, 4) ||
        !aligned_to(num_accepted, 4) || (seq_status && !aligned_to(seq_status, 4)))
        return SV_ERR_ALIGN;
    if ((lse_t && !aligned_to(lse_t, 8)) || (lse_d && !aligned_to(lse_d, 8)) ||
        (log_ratio && !aligned_to(log_ratio, 8)))
        return SV_ERR_ALIGN;
    if (!aligned_to(workspace, kAlign)) return SV_ERR_WORKSPACE;
    Geometry g;
    LmLayout L;
    rc = lm_plan(B, K, V, Dt, Dd, mode, &g, &L);
    if (rc != SV_OK) return rc;
    if (workspace_bytes < L.total) return SV_ERR_WORKSPACE;
    g.pdl = 0;  // the scan reads the token logits as soon as it starts
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto* part = reinterpret_cast<sv::Partial*>(ws + L.part);
    auto* tok = reinterpret_cast<float*>(ws + L.tok);
    auto* seqs = reinterpret_cast<sv::SeqRecord*>(ws + L.seqs);
    auto* err = reinterpret_cast<int32_t*>(ws + L.err);

    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
    sv::LmArgs la{};
    la.p[0] = sv::LmProblem{hidden_t, w_t, B * (K + 1), Dt, 0, static_cast<int32_t>(K + 1),
                            nullptr, 0, 0, 0, 0};
    la.nprob = 1;
    if (with_draft) {
        la.p[1] = sv::LmProblem{hidden_d, w_d, B * K, Dd, B * (K + 1), static_cast<int32_t>(K),
                                nullptr, 0, 0, 0, 0};
        la.nprob = 2;
    }
    la.V = V;
    la.K = static_cast<int32_t>(K);
    la.tokens = tokens;
    la.c = c;
    la.greedy = sampling ? 0 : 1;
    la.part = part;
    la.tok = tok;
    la.err = err;
    la.gate = gate;
    bool mapped = false;
    if (!record(0)) return SV_ERR_CUDA;
    if (sv::launch_lmhead(sv::kLmStats, la, s, &mapped) != cudaSuccess || !mapped)
        return SV_ERR_CUDA;
    if (!record(1)) return SV_ERR_CUDA;

    const sv::RowMap full{nullptr, nullptr, 0, static_cast<int32_t>(K + 1),
                          static_cast<int32_t>(sampling ? K : 0)};
    sv::ScanArgs sa{};
    sa.tokens = tokens;
    sa.g = g;
    sa.c = c;
    sa.seed = seed;
    sa.partials = part;
    sa.out_tokens = out_tokens;
    sa.num_accepted = num_accepted;
    sa.seqs = seqs;
    sa.lse_t = sampling ? lse_t : nullptr;
    sa.lse_d = sampling ? lse_d : nullptr;
    sa.log_ratio = sampling ? log_ratio : nullptr;
    sa.seq_status = seq_status;
    sa.map = full;
    sa.lm_tiles = L.n_vt;
    sa.tok = sampling ? tok : nullptr;
    if (sv::launch_scan(sa, s) != cudaSuccess) return SV_ERR_CUDA;
    if (!record(2)) return SV_ERR_CUDA;

    if (sampling) {
        // The emitted pair of every sequence: hidden states gathered, then
        // their logits [B][2][V] (target row, draft row) as float32.
        uint8_t* ht = ws + L.ht;
        uint8_t* hd = ws + L.hd;
        float* pairs = reinterpret_cast<float*>(ws + L.pairs);
        if (sv::launch_gather_hidden(hidden_t, with_draft ? hidden_d : nullptr, seqs, B, K, Dt,
                                     with_draft ? Dd : 0, ht, hd, s) != cudaSuccess)
            return SV_ERR_CUDA;
        sv::LmArgs le{};
        le.p[0] = sv::LmProblem{ht, w_t, B, Dt, 0, 0, pairs, 2 * V, 0, 0, 0};
        le.nprob = 1;
        if (with_draft) {
            le.p[1] = sv::LmProblem{hd, w_d, B, Dd, 0, 0, pairs + V, 2 * V, 0, 0, 0};
            le.nprob = 2;
        }
        le.V = V;
        le.err = err;
        if (sv::launch_lmhead(sv::kLmLogits, le, s, &mapped) != cudaSuccess || !mapped)
            return SV_ERR_CUDA;
        if (!record(3)) return SV_ERR_CUDA;
        const int64_t row_bytes = V * 4;
        const uint8_t* pb = reinterpret_cast<const uint8_t*>(pairs);
        sv::RowPairLayout lay{2, 0, 2, 0, pb + 2 * B * row_bytes, pb + 2 * B * row_bytes};
        sv::SampleArgs pa{pb, pb + row_bytes, g, c, seed, seqs,
                          reinterpret_cast<float*>(ws + L.block_sums), out_tokens, num_accepted,
                          seq_status, lay, 0, sv::Shards{}, 0};
        if (sv::launch_sample(pa, s) != cudaSuccess) return SV_ERR_CUDA;
    } else if (!record(3)) {
        return SV_ERR_CUDA;
    }
    if (sv::launch_lm_fail(err, B, K, out_tokens, num_accepted, seq_status, s) != cudaSuccess)
        return SV_ERR_CUDA;
    if (!record(4)) return SV_ERR_CUDA;
    return SV_OK;
}

}  // namespace

SV_EXPORT int sv_lmhead_workspace_bytes(int64_t B, int64_t K, int64_t V, int64_t d_target,
                                        int64_t d_draft, int mode, size_t* bytes)
{
    if (bytes == nullptr) return SV_ERR_ARG;
    Geometry g;
    LmLayout L;
    const int rc = lm_plan(B, K, V, d_target, d_draft, mode, &g, &L);
    if (rc != SV_OK) return rc;
    *bytes = L.total;
    return SV_OK;
}

SV_EXPORT int spec_verify_lmhead(const void* hidden_target, const void* weight_target,
                                 const void* hidden_draft, const void* weight_draft,
                                 const int32_t* draft_tokens, int64_t B, int64_t K, int64_t V,
                                 int64_t d_target, int64_t d_draft, float temperature,
                                 uint64_t seed, int mode, int32_t* out_tokens,
                                 int32_t* num_accepted, void* workspace, size_t workspace_bytes,
                                 void* stream)
{
    return run_lmhead(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens, B, K,
                      V, d_target, d_draft, temperature, seed, mode, out_tokens, num_accepted,
                      workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr,
                      nullptr, 0);
}

SV_EXPORT int spec_verify_lmhead_debug(const void* hidden_target, const void* weight_target,
                                       const void* hidden_draft, const void* weight_draft,
                                       const int32_t* draft_tokens, int64_t B, int64_t K,
                                       int64_t V, int64_t d_target, int64_t d_draft,
                                       float temperature, uint64_t seed, int mode,
                                       int32_t* out_tokens, int32_t* num_accepted,
                                       void* workspace, size_t workspace_bytes, void* stream,
                                       double* lse_t, double* lse_d, double* log_ratio,
                                       int32_t* seq_status)
{
    return run_lmhead(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens, B, K,
                      V, d_target, d_draft, temperature, seed, mode, out_tokens, num_accepted,
                      workspace, workspace_bytes, stream, lse_t, lse_d, log_ratio, seq_status,
                      nullptr, 0);
}

SV_EXPORT int spec_verify_lmhead_timed(const void* hidden_target, const void* weight_target,
                                       const void* hidden_draft, const void* weight_draft,
                                       const int32_t* draft_tokens, int64_t B, int64_t K,
                                       int64_t V, int64_t d_target, int64_t d_draft,
                                       float temperature, uint64_t seed, int mode,
                                       int32_t* out_tokens, int32_t* num_accepted,
                                       void* workspace, size_t workspace_bytes, void* stream,
                                       void* const* events, int n_events)
{
    if (events == nullptr) return SV_ERR_ARG;
    return run_lmhead(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens, B, K,
                      V, d_target, d_draft, temperature, seed, mode, out_tokens, num_accepted,
                      workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr,
                      events, n_events);
}

SV_EXPORT int spec_verify_lmhead_gated(const void* hidden_target, const void* weight_target,
                                       const void* hidden_draft, const void* weight_draft,
                                       const int32_t* draft_tokens, int64_t B, int64_t K,
                                       int64_t V, int64_t d_target, int64_t d_draft,
                                       float temperature, uint64_t seed, int mode,
                                       int32_t* out_tokens, int32_t* num_accepted,
                                       void* workspace, size_t workspace_bytes, void* stream,
                                       int32_t* seq_status, const int32_t* gate)
{
    if (gate == nullptr) return SV_ERR_ARG;
    if (!aligned_to(gate, 4)) return SV_ERR_ALIGN;
    return run_lmhead(hidden_target, weight_target, hidden_draft, weight_draft, draft_tokens, B, K,
                      V, d_target, d_draft, temperature, seed, mode, out_tokens, num_accepted,
                      workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, seq_status,
                      nullptr, 0, gate);
}

SV_EXPORT int sv_lmhead_logits(const void* hidden, const void* weight, int64_t R, int64_t D,
                               int64_t V, float* out, int32_t* err, void* stream)
{
    if (R < 0 || V < 1 || D < 8 || D % 8 != 0) return SV_ERR_ARG;
    if (R >= (int64_t(1) << 31) || V >= (int64_t(1) << 31) || D >= (int64_t(1) << 31))
        return SV_ERR_SIZE;
    if (R == 0) return SV_OK;
    if (hidden == nullptr || weight == nullptr || out == nullptr || err == nullptr)
        return SV_ERR_ARG;
    if (!aligned_to(hidden, 16) || !aligned_to(weight, 16) || !aligned_to(out, 4) ||
        !aligned_to(err, 4))
        return SV_ERR_ALIGN;
    sv::LmArgs la{};
    la.p[0] = sv::LmProblem{hidden, weight, R, D, 0, 0, out, V, 0, 0, 0};
    la.nprob = 1;
    la.V = V;
    la.err = err;
    bool mapped = false;
    if (sv::launch_lmhead(sv::kLmLogits, la, static_cast<cudaStream_t>(stream), &mapped) !=
            cudaSuccess ||
        !mapped)
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

SV_EXPORT int sv_version(void) { return 105; }

SV_EXPORT int sv_device_checks(void)
{
#ifdef SV_DEVICE_CHECKS
    return 1;
#else
    return 0;
#endif
}
