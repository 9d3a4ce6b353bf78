// qh_api.cu -- the C ABI of include/qhead.h: argument checks, the launch plan,
// workspace layout and the kernel sequence of each entry point.
//
// Forward sequence:  compact (mask -> active rows) -> convert (bf16 -> fp16 rows)
//                    -> head kernel (per-split partials) -> finalize (merge,
//                    exact target logit, argmax recheck, scatter).
// Backward sequence: compact -> head backward (per-split partial dh) ->
//                    finalize (fixed-order sum, exact one-hot term, zeros for
//                    masked rows).
#include <stdio.h>

#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/qhead.h"
#include "qh_internal.cuh"
#include "qh_tmap.h"

static_assert(QHEAD_SB_F16 == qh::kSbF16 && QHEAD_SB_BF16 == qh::kSbBf16 &&
                  QHEAD_SB_F32 == qh::kSbF32,
              "scale/bias element type codes");

namespace {

thread_local std::string g_err;
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;
thread_local bool g_stall = false;

// Consumes the one-shot stall switch of qhead_test_stall_next_call.
int take_stall() {
    const bool s = g_stall;
    g_stall = false;
    return s ? 1 : 0;
}

// Records the armed "before head kernel" event (if any).
void hook_before(cudaStream_t st) {
    if (g_ev_start) cudaEventRecord(g_ev_start, st);
}
void hook_after(cudaStream_t st) {
    if (g_ev_stop) cudaEventRecord(g_ev_stop, st);
    g_ev_start = g_ev_stop = nullptr;
}

// Disarms both one-shot hooks when the entry point that holds it returns, so
// that a call rejected before its kernels ran does not leave them armed for
// the thread's next call.
struct HookScope {
    ~HookScope() {
        g_ev_start = g_ev_stop = nullptr;
        g_stall = false;
    }
};

int fail(int code, const std::string& msg) {
    g_err = msg;
    return code;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// The caller's scales and biases in their own type (the exact fp32 parts).
qh::SbView sb_view(const qhead_head* hd) { return qh::SbView{hd->scales, hd->biases, hd->sb_dtype}; }

struct DevInfo {
    int sms = 0;
};

int device_info(DevInfo* info) {
    info->sms = qh::device_sms();
    if (info->sms <= 0) return fail(QHEAD_ECUDA, "cannot query the current device's SM count");
    return QHEAD_OK;
}

int check_head(const qhead_head* hd) {
    if (!hd) return fail(QHEAD_EINVAL, "head is NULL");
    if (!hd->wq || !hd->scales || !hd->biases) return fail(QHEAD_EINVAL, "head pointer is NULL");
    if (hd->bits != 4 && hd->bits != 8) return fail(QHEAD_EUNSUPPORTED, "bits must be 4 or 8");
    if (hd->group != 64) return fail(QHEAD_EUNSUPPORTED, "group size must be 64");
    if (hd->sb_dtype != QHEAD_SB_F16 && hd->sb_dtype != QHEAD_SB_BF16 &&
        hd->sb_dtype != QHEAD_SB_F32)
        return fail(QHEAD_EUNSUPPORTED, "sb_dtype must be QHEAD_SB_F16, QHEAD_SB_BF16 or QHEAD_SB_F32");
    if (hd->H < 128 || hd->H > qh::kMaxH || hd->H % 128)
        return fail(QHEAD_EUNSUPPORTED, "H must be a multiple of 128 in [128, 8192]");
    if (hd->V < 1 || hd->V >= ((int64_t)1 << 31)) return fail(QHEAD_EINVAL, "V must be in [1, 2^31)");
    if (reinterpret_cast<uintptr_t>(hd->wq) % 16) return fail(QHEAD_EINVAL, "wq must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(hd->scales) % 16 || reinterpret_cast<uintptr_t>(hd->biases) % 16)
        return fail(QHEAD_EINVAL, "scales/biases must be 16-byte aligned");
    if (hd->softcap != hd->softcap) return fail(QHEAD_EINVAL, "softcap is NaN");
    return QHEAD_OK;
}

// ---------------------------------------------------------------- plans

// Workspace for the fp16 copies of a bf16 / fp32 head's scales and biases
// (two [V, H/64] arrays, each 256-byte aligned); none for an fp16 head.
size_t sb_copy_bytes(const qhead_head* hd) {
    if (hd->sb_dtype == QHEAD_SB_F16) return 0;
    return 2 * align_up(2 * (size_t)hd->V * (size_t)(hd->H / 64), 256);
}

// The scales and biases the kernels with fp16 operands read: the caller's
// arrays for an fp16 head, else their fp16 copies in the workspace region at
// `off`, written by a conversion launch on `st` (which this queues).
int sb_operands(const qhead_head* hd, void* ws, size_t off, cudaStream_t st, const __half** sc,
                const __half** bi) {
    if (hd->sb_dtype == QHEAD_SB_F16) {
        *sc = static_cast<const __half*>(hd->scales);
        *bi = static_cast<const __half*>(hd->biases);
        return QHEAD_OK;
    }
    const size_t n = (size_t)hd->V * (size_t)(hd->H / 64);
    __half* s16 = at<__half>(ws, off);
    __half* b16 = at<__half>(ws, off + align_up(2 * n, 256));
    const cudaError_t e = qh::launch_sb_to_f16(sb_view(hd), (int64_t)n, s16, b16, st);
    if (e) return fail(QHEAD_ECUDA, std::string("sb_to_f16: ") + cudaGetErrorString(e));
    *sc = s16;
    *bi = b16;
    return QHEAD_OK;
}

// Rows from which the forward runs on the tensor-core kernel (below: the
// weight-streaming kernel, whose cost is one pass over the head per 8 rows).
// Measured on the Gemma-class head (V = 262144, H = 2560, 4-bit): the
// streaming forward takes 0.084 ms at 1-8 rows and 0.14 ms at 16, the
// tensor-core forward 0.27-0.28 ms from 1 to 128 rows; from 17 rows (three
// token groups) the streaming kernel is the slower one (0.36 ms at 24, 0.47
// at 63).  The backward always runs on the tensor cores (0.49-0.52 ms from
// 1 to 128 rows; the CUDA-core backward it replaced took 7.7 ms at 1-8 rows
// and 56 ms at 63).
constexpr int64_t kTcMinFwdM = 17;

struct FwdPlan {
    int64_t M = 0, Mpad = 0;
    bool tc = false;     // tensor-core path
    int grid = 0;        // persistent CTAs of the tensor-core kernel
    int S = 1;           // vocab splits of the partials (weight-streaming path)
    size_t records = 0;  // partial records
    size_t off_count = 0, off_rows = 0, off_pos = 0, off_h16 = 0, off_part = 0, total = 0;
    size_t off_sb = 0;   // fp16 copies of bf16 / fp32 scales and biases (else unused)
};

struct BwdPlan {
    int64_t M = 0, Mpad = 0;
    int grid = 0;
    int S = 1;               // K slices of the dh contraction
    int64_t chunk = 0;       // vocab rows per coefficient block (tensor-core path)
    bool dw = false;         // head gradient requested: the regions below are planned
    bool skip = false;       // blockMax early exit: the skip map is planned
    bool filter = false;     // coefficient filter: the dh step bits are planned
    int64_t n_vt = 0;        // vocab tiles of 256 rows
    int64_t kbits_ld = 0;    // filter: 64-bit words of vocab-step bits per 256-row unit
    size_t off_count = 0, off_rows = 0, off_pos = 0, off_h16 = 0, off_coeff = 0, off_dhp = 0,
           off_hp = 0, off_g = 0, off_dmax = 0, off_cnt = 0, off_offs = 0, off_cursor = 0,
           off_idx = 0, off_skip = 0, off_kbits = 0, total = 0;
    size_t off_sb = 0;       // fp16 copies of bf16 / fp32 scales and biases (else unused)
};

// Vocab rows per backward chunk: the [rows x chunk] fp16 coefficient block is
// sized up to 4 GiB of workspace, so that the 8192-row workloads run the
// whole vocabulary as one chunk (3 GB at 5736 active rows x 262144): the dh
// contraction then accumulates each output tile over the entire vocabulary
// in tensor memory and writes its K-slice partials once, instead of adding
// them into dh after every chunk.  Measured on the masked 8192-row Gemma
// workload: backward 11.9 ms with 96 MB chunks (16 chunks), 11.4 ms with
// 384 MB, 10.8 ms with 1 GiB, 10.5 ms with one chunk; 7.0 vs 7.6 ms per step
// on the 8-bit head.  Larger heads or row counts fall back to chunks of at
// least 16384 rows.
constexpr int64_t kBwdCoeffBudget = (int64_t)4 << 30;
constexpr int64_t kBwdChunkMin = 16384;
constexpr int64_t kBwdSkipChunkMin = 65536;

// K slices of the dh contraction: enough (m, n) tiles x slices to fill the
// SMs in whole waves (each slice accumulates into its own buffer).
int dh_slices(int64_t Mpad, int H, int sms, int64_t n_k_min) {
    const int64_t tiles = ((Mpad + 255) / 256) * (H / qh::tc_dh_cols(H));  // 256-row units
    int best = 1;
    double best_eff = 0.0;
    for (int ks = 1; ks <= 16 && ks <= n_k_min; ++ks) {
        const int64_t units = tiles * ks;
        const int64_t waves = (units + sms - 1) / sms;
        const double eff = (double)units / (double)(waves * sms);
        if (eff > best_eff + 0.02) { best_eff = eff; best = ks; }
        if (eff >= 0.9 && waves >= 2) break;
    }
    return best;
}

// force_tc: the tensor-core path for every M (the per-tile maxima of the
// blockMax early exit come from its epilogue).
int plan_fwd(const qhead_head* hd, int64_t M, FwdPlan* p, bool force_tc = false) {
    DevInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    p->M = M;
    p->Mpad = (M + qh::kRowPad - 1) / qh::kRowPad * qh::kRowPad;
    p->tc = M >= kTcMinFwdM || force_tc;
    if (p->tc) {
        // One persistent CTA per SM; the kernel picks the number of vocab
        // segments S from the active-row count so that n_tiles * S is about
        // 32 * grid, hence at most 128 * (32 * grid + n_tiles) records.
        // Partial records: the kernel writes record i * S + s for compact
        // rows i < the active count and vocab segments s < S, where S is at
        // most the number of 256-row vocab tiles and S * (256-row units) is
        // about 32 per CTA pair; either bound caps the records.
        p->grid = di.sms;
        const size_t n_vt = (size_t)((hd->V + 255) / 256);
        const size_t by_rows = (size_t)p->Mpad * n_vt;
        const size_t by_units = (size_t)128 * (32 * (size_t)p->grid + (size_t)(p->Mpad / 128));
        p->records = by_rows < by_units ? by_rows : by_units;
    } else {
        const int64_t groups = (M + qh::kTokGroup - 1) / qh::kTokGroup;
        // One full wave: every SM holds as many CTAs as fit; each split keeps at
        // least one 256-row tile (16 rows per consumer warp).
        const int64_t want = (int64_t)di.sms * qh::stream_fwd_ctas_per_sm(hd->bits, hd->H);
        int64_t S = (want + groups - 1) / groups;
        const int64_t max_s = (hd->V + 255) / 256;
        if (S > max_s) S = max_s;
        if (S < 1) S = 1;
        p->S = (int)S;
        p->records = (size_t)p->Mpad * p->S;
    }
    size_t off = 0;
    p->off_count = off; off = align_up(off + 16, 256);  // count, error word, segment count
    p->off_rows = off;  off = align_up(off + 4 * (size_t)p->Mpad, 256);
    p->off_pos = off;   off = align_up(off + 4 * (size_t)M, 256);
    // fp16 h for the tensor-core path; the streaming kernel converts its rows itself.
    p->off_h16 = off;   if (p->tc) off = align_up(off + 2 * (size_t)p->Mpad * hd->H, 1024);
    p->off_part = off;  off = align_up(off + sizeof(qh::Partial) * p->records, 256);
    p->off_sb = off;    off += sb_copy_bytes(hd);
    p->total = off;
    return QHEAD_OK;
}

// with_dw: the head gradient is requested too; it reuses the tensor-core
// path's coefficient blocks.  with_skip: the blockMax early exit, whose skip
// map is in the tensor-core kernels' tiles.  with_filter: the coefficient
// filter, decided in the tensor-core coefficient epilogue.  Each takes that
// path for every M.
int plan_bwd(const qhead_head* hd, int64_t M, BwdPlan* p, bool with_dw = false,
             bool with_skip = false, bool with_filter = false) {
    DevInfo di;
    int rc = device_info(&di);
    if (rc) return rc;
    p->M = M;
    p->Mpad = (M + qh::kRowPad - 1) / qh::kRowPad * qh::kRowPad;
    p->dw = with_dw;
    p->skip = with_skip;
    p->filter = with_filter;
    p->n_vt = (hd->V + qh::kTcFwdTileRows - 1) / qh::kTcFwdTileRows;
    size_t off = 0;
    p->off_count = off; off = align_up(off + 16, 256);
    p->off_rows = off;  off = align_up(off + 4 * (size_t)p->Mpad, 256);
    p->off_pos = off;   off = align_up(off + 4 * (size_t)M, 1024);
    // (dh_slices is declared above plan_fwd)
    p->grid = di.sms;
    p->S = 1;
    // Vocab rows rounded to the logit kernel's tiles; the slice count S is
    // kept within the K steps of the shortest (last) chunk, so every chunk
    // writes or adds every slice.
    const int64_t tr = qh::kTcFwdTileRows;
    const int64_t vr = (hd->V + tr - 1) / tr * tr;
    int64_t chunk = kBwdCoeffBudget / (2 * p->Mpad) / 256 * 256;
    if (chunk < kBwdChunkMin) chunk = kBwdChunkMin;
    // With the blockMax early exit most tiles are skipped: fewer, longer
    // chunks (fewer launches of mostly empty kernels) pay more than L2
    // residency (measured 4.69 -> 3.28 ms per call at 8192 peaked rows).
    if (with_skip && chunk < kBwdSkipChunkMin) chunk = kBwdSkipChunkMin;
    if (chunk > vr) chunk = vr;
    p->chunk = chunk;
    const int64_t last = vr - (vr - 1) / chunk * chunk;  // rows of the last chunk
    p->S = dh_slices(p->Mpad, hd->H, p->grid, (last < chunk ? last : chunk) / 64);
    p->off_h16 = off;   off = align_up(off + 2 * (size_t)p->Mpad * hd->H, 1024);
    p->off_coeff = off; off = align_up(off + 2 * (size_t)p->Mpad * p->chunk, 1024);
    p->off_dhp = off;   off = align_up(off + 4 * (size_t)p->S * p->Mpad * hd->H, 1024);
    if (with_dw) {
        p->off_hp = off;     off = align_up(off + 2 * (size_t)p->Mpad * hd->H, 1024);
        p->off_g = off;      off = align_up(off + 4 * (size_t)p->Mpad, 256);
        p->off_dmax = off;   off = align_up(off + 16, 256);
        p->off_cnt = off;    off = align_up(off + 4 * (size_t)hd->V, 256);
        p->off_offs = off;   off = align_up(off + 4 * ((size_t)hd->V + 1), 256);
        p->off_cursor = off; off = align_up(off + 4 * (size_t)hd->V, 256);
        p->off_idx = off;    off = align_up(off + 4 * (size_t)p->Mpad, 256);
    }
    if (with_skip) {
        p->off_skip = off;   off = align_up(off + (size_t)(p->Mpad / 128) * p->n_vt, 256);
    }
    if (with_filter) {
        // one bit per (256-row dh unit, 64-row vocab step of the head)
        p->kbits_ld = (p->n_vt * 4 + 63) / 64;
        p->off_kbits = off;
        off = align_up(off + 8 * (size_t)((p->Mpad + 255) / 256) * p->kbits_ld, 256);
    }
    off = align_up(off, 256);
    p->off_sb = off;    off += sb_copy_bytes(hd);
    p->total = off;
    return QHEAD_OK;
}


int cuda_fail(cudaError_t e, const char* what) {
    return fail(QHEAD_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace

void qh::set_error(const std::string& msg) { g_err = msg; }

extern "C" {

const char* qhead_last_error(void) { return g_err.c_str(); }

const char* qhead_version(void) { return "qhead 0.1.0 sm_103a"; }

void qhead_test_stall_next_call(int armed) { g_stall = armed != 0; }

void qhead_time_next_head_kernel(void* start, void* stop) {
    g_ev_start = static_cast<cudaEvent_t>(start);
    g_ev_stop = static_cast<cudaEvent_t>(stop);
}

size_t qhead_fwd_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    FwdPlan p;
    if (plan_fwd(head, M, &p)) return (size_t)-1;
    return p.total;
}

size_t qhead_bwd_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    BwdPlan p;
    if (plan_bwd(head, M, &p)) return (size_t)-1;
    return p.total;
}

size_t qhead_fwd_blockmax_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    FwdPlan p;
    if (plan_fwd(head, M, &p, true)) return (size_t)-1;
    return p.total;
}

// The forward; bmax != NULL also writes the per-tile maxima of z (and takes
// the tensor-core path).
static int fwd_impl(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                    const uint8_t* mask, float* logp, float* lse, int32_t* argmax, float* bmax,
                    void* workspace, size_t workspace_bytes, void* stream) {
    HookScope hooks;
    g_err.clear();
    const int stall = take_stall();
    int rc = check_head(head);
    if (rc) return rc;
    if (M < 0) return fail(QHEAD_EINVAL, "M < 0");
    if (M >= ((int64_t)1 << 31) - qh::kRowPad) return fail(QHEAD_EINVAL, "M too large");
    if (M == 0) return QHEAD_OK;
    if (!h) return fail(QHEAD_EINVAL, "h is NULL");
    if (reinterpret_cast<uintptr_t>(h) % 16) return fail(QHEAD_EINVAL, "h must be 16-byte aligned");
    if (logp && !targets) return fail(QHEAD_EINVAL, "logp requested without targets");
    if (!logp && !lse && !argmax && !bmax) return fail(QHEAD_EINVAL, "no output requested");
    if (!workspace) return fail(QHEAD_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(QHEAD_EINVAL, "workspace must be 256-byte aligned");
    if (bmax && reinterpret_cast<uintptr_t>(bmax) % 4)
        return fail(QHEAD_EINVAL, "block_max must be 4-byte aligned");
    FwdPlan p;
    rc = plan_fwd(head, M, &p, bmax != nullptr);
    if (rc) return rc;
    if (workspace_bytes < p.total)
        return fail(QHEAD_EINVAL, "workspace too small: need " + std::to_string(p.total) + " bytes");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* wq = head->wq;
    const __half *sc = nullptr, *bi = nullptr;
    if ((rc = sb_operands(head, workspace, p.off_sb, st, &sc, &bi))) return rc;
    const qh::SbView sbx = sb_view(head);
    const auto* hb = static_cast<const __nv_bfloat16*>(h);
    int* count = at<int>(workspace, p.off_count);
    int* err = count + 1;
    int* S_dev = count + 2;
    int* rows = at<int>(workspace, p.off_rows);
    int* pos = at<int>(workspace, p.off_pos);
    __half* h16 = at<__half>(workspace, p.off_h16);
    qh::Partial* part = at<qh::Partial>(workspace, p.off_part);

    cudaError_t e;
    if (p.tc) {
        if (M <= qh::kFusedPrologueMaxM) {
            if ((e = qh::launch_prologue_fused(mask, hb, M, p.Mpad, head->H, head->bits, rows, pos,
                                               count, h16, p.Mpad, err, st)))
                return cuda_fail(e, "prologue");
        } else {
            if ((e = qh::launch_compact(mask, M, p.Mpad, rows, pos, count, err, st)))
                return cuda_fail(e, "compact");
            if ((e = qh::launch_convert_h(hb, p.Mpad, head->H, head->bits, rows, count, h16, st)))
                return cuda_fail(e, "convert_h");
        }
        CUtensorMap th, tw;
        const int words = 64 * head->bits / 32;
        if (!qh::tmap_rows_f16_sw128(&th, h16, head->H, p.Mpad, 128) ||
            !qh::tmap_packed_rows(&tw, wq, head->H * head->bits / 32, head->V, words,
                                  qh::kTcFwdBoxRows))
            return fail(QHEAD_ECUDA, "TMA tensor map encoding failed");
        qh::TcFwdArgs ta{};
        ta.scales = sc; ta.biases = bi; ta.V = head->V; ta.H = head->H; ta.cap = head->softcap;
        ta.count = count; ta.err = err; ta.stall = stall;
        ta.vt_begin = 0; ta.vt_end = (int)((head->V + qh::kTcFwdTileRows - 1) / qh::kTcFwdTileRows);
        ta.part = part; ta.S_out = S_dev;
        if (bmax) {
            ta.bmax = bmax;
            ta.bmax_ld = ta.vt_end;  // vocab tiles of 256 rows
            ta.rows = rows;
        }
        hook_before(st);
        e = qh::launch_tc_fwd(th, tw, ta, head->bits, false, p.grid, st);
        hook_after(st);
        if (e) return cuda_fail(e, "tc_fwd");
    } else {
        hook_before(st);
        // Compaction, fp16 conversion and group sums happen inside this kernel.
        e = qh::launch_stream_fwd(wq, sc, bi, head->V, head->H, head->bits, head->softcap, hb,
                                  mask, M, rows, pos, count, part, p.S, err, stall, st);
        hook_after(st);
        if (e) return cuda_fail(e, "stream_fwd");
    }
    if ((e = qh::launch_fwd_finalize(wq, sbx, head->V, head->H, head->bits, head->softcap, hb,
                                     pos, targets, part, p.S, p.tc ? S_dev : nullptr, err,
                                     logp, lse, argmax, M, st)))
        return cuda_fail(e, "fwd_finalize");
    return QHEAD_OK;
}

size_t qhead_bwd_dw_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    BwdPlan p;
    if (plan_bwd(head, M, &p, true)) return (size_t)-1;
    return p.total;
}

// The backward chain: dh (if dh != NULL) and the head gradient (if dw != NULL).
static int bwd_impl(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                    const uint8_t* mask, const float* lse, const float* dlogp, float* dh,
                    float* dw, const float* bmax, float eps, bool filter, uint8_t* cold_out,
                    void* workspace, size_t workspace_bytes, void* stream) {
    HookScope hooks;
    g_err.clear();
    const int stall = take_stall();
    int rc = check_head(head);
    if (rc) return rc;
    if (M < 0) return fail(QHEAD_EINVAL, "M < 0");
    if (M >= ((int64_t)1 << 31) - qh::kRowPad) return fail(QHEAD_EINVAL, "M too large");
    if (M == 0 && !dw) return QHEAD_OK;
    if (!dh && !dw) return fail(QHEAD_EINVAL, "dh (or, in qhead_bwd_dw, dw) is required");
    if (dw && reinterpret_cast<uintptr_t>(dw) % 32)
        return fail(QHEAD_EINVAL, "dw must be 32-byte aligned");
    if (M == 0) {  // no rows: nothing for dh; the head gradient is zero
        if (!dw) return QHEAD_OK;
        cudaError_t e = cudaMemsetAsync(dw, 0, sizeof(float) * (size_t)head->V * head->H,
                                        static_cast<cudaStream_t>(stream));
        return e ? cuda_fail(e, "dw zero") : QHEAD_OK;
    }
    if (!h || !targets || !lse || !dlogp)
        return fail(QHEAD_EINVAL, "h, targets, lse and dlogp are required");
    if (reinterpret_cast<uintptr_t>(h) % 16) return fail(QHEAD_EINVAL, "h must be 16-byte aligned");
    if (dh && reinterpret_cast<uintptr_t>(dh) % 16)
        return fail(QHEAD_EINVAL, "dh must be 16-byte aligned");
    if (!workspace) return fail(QHEAD_EINVAL, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(QHEAD_EINVAL, "workspace must be 256-byte aligned");
    BwdPlan p;
    rc = plan_bwd(head, M, &p, dw != nullptr, bmax != nullptr, filter);
    if (rc) return rc;
    if (workspace_bytes < p.total)
        return fail(QHEAD_EINVAL, "workspace too small: need " + std::to_string(p.total) + " bytes");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* wq = head->wq;
    const __half *sc = nullptr, *bi = nullptr;
    if ((rc = sb_operands(head, workspace, p.off_sb, st, &sc, &bi))) return rc;
    const qh::SbView sbx = sb_view(head);
    const auto* hb = static_cast<const __nv_bfloat16*>(h);
    int* count = at<int>(workspace, p.off_count);
    int* err = count + 1;
    int* rows = at<int>(workspace, p.off_rows);
    int* pos = at<int>(workspace, p.off_pos);
    float* dhp = at<float>(workspace, p.off_dhp);

    cudaError_t e;
    __half* h16 = at<__half>(workspace, p.off_h16);
    __half* coeff = at<__half>(workspace, p.off_coeff);
    if (M <= qh::kFusedPrologueMaxM) {
        if ((e = qh::launch_prologue_fused(mask, hb, M, p.Mpad, head->H, head->bits, rows, pos,
                                           count, h16, p.Mpad, err, st)))
            return cuda_fail(e, "prologue");
    } else {
        if ((e = qh::launch_compact(mask, M, p.Mpad, rows, pos, count, err, st)))
            return cuda_fail(e, "compact");
        if ((e = qh::launch_convert_h(hb, p.Mpad, head->H, head->bits, rows, count, h16, st)))
            return cuda_fail(e, "convert_h");
    }
    // blockMax early exit: the (row tile, vocab tile) pairs both phases skip.
    uint8_t* skip = p.skip ? at<uint8_t>(workspace, p.off_skip) : nullptr;
    if (skip && (e = qh::launch_skip_map(bmax, p.n_vt, lse, targets, rows, count, p.Mpad / 128,
                                         p.n_vt, eps, skip, st)))
        return cuda_fail(e, "skip_map");
    // Coefficient filter: every dh step starts skipped and every block cold
    // (rows past the active ones stay so); the coefficient pass clears the
    // bits of the steps that hold a warm block.
    auto* kbits = p.filter ? at<unsigned long long>(workspace, p.off_kbits) : nullptr;
    const int64_t n_vb = (head->V + 31) / 32, n_rb = (M + 31) / 32;
    if (kbits && (e = cudaMemsetAsync(kbits, 0xff,
                                      8 * (size_t)((p.Mpad + 255) / 256) * p.kbits_ld, st)))
        return cuda_fail(e, "filter bits");
    if (kbits && cold_out && (e = cudaMemsetAsync(cold_out, 1, (size_t)(n_rb * n_vb), st)))
        return cuda_fail(e, "cold output");
    // Head gradient: max |dlogp|, the scaled fp16 h', the one-hot terms and
    // the per-target row lists, once per call.
    __half* hp = p.dw ? at<__half>(workspace, p.off_hp) : nullptr;
    float* g = p.dw ? at<float>(workspace, p.off_g) : nullptr;
    float* dmax = p.dw ? at<float>(workspace, p.off_dmax) : nullptr;
    int* offs = p.dw ? at<int>(workspace, p.off_offs) : nullptr;
    int* idx = p.dw ? at<int>(workspace, p.off_idx) : nullptr;
    if (p.dw &&
        (e = qh::launch_dw_prep(wq, sbx, head->V, head->H, head->bits, head->softcap, hb,
                                rows, count, targets, dlogp, p.Mpad, dmax, hp, g,
                                at<int>(workspace, p.off_cnt), offs,
                                at<int>(workspace, p.off_cursor), idx, st)))
        return cuda_fail(e, "dw_prep");
    CUtensorMap th, tw_logit, tcoef, tw_dh, tcoef_t{}, thp{};
    if (p.dw && (!qh::tmap_rows_f16_sw128(&tcoef_t, at<__half>(workspace, p.off_coeff),
                                           p.chunk, p.Mpad, 64) ||
                 !qh::tmap_rows_f16_sw128(&thp, hp, head->H, p.Mpad, 64)))
        return fail(QHEAD_ECUDA, "TMA tensor map encoding failed");
    const int wpr = head->H * head->bits / 32;
    if (!qh::tmap_rows_f16_sw128(&th, h16, head->H, p.Mpad, 128) ||
        !qh::tmap_packed_rows(&tw_logit, wq, wpr, head->V, 64 * head->bits / 32,
                              qh::kTcFwdBoxRows) ||
        !qh::tmap_rows_f16_sw128(&tcoef, coeff, p.chunk, p.Mpad, 128) ||
        !(qh::tc_dh_swizzled(head->H, head->bits)
              ? qh::tmap_packed_rows_sw128(&tw_dh, wq, wpr, head->V, 64)
              : qh::tmap_packed_rows(&tw_dh, wq, wpr, head->V,
                                     qh::tc_dh_words(head->H, head->bits), 64)))
        return fail(QHEAD_ECUDA, "TMA tensor map encoding failed");
    const int tr = qh::kTcFwdTileRows;
    const int n_vt = (int)((head->V + tr - 1) / tr);
    const int vt_chunk = (int)(p.chunk / tr);
    hook_before(st);
    for (int vt0 = 0, c = 0; vt0 < n_vt; vt0 += vt_chunk, ++c) {
        const int vt1 = vt0 + vt_chunk < n_vt ? vt0 + vt_chunk : n_vt;
        qh::TcFwdArgs ta{};
        ta.scales = sc; ta.biases = bi; ta.V = head->V; ta.H = head->H;
        ta.cap = head->softcap; ta.count = count; ta.err = err;
        ta.stall = vt0 == 0 ? stall : 0;
        ta.vt_begin = vt0; ta.vt_end = vt1;
        ta.lse = lse; ta.rows = rows; ta.coeff = coeff; ta.coeff_ld = p.chunk;
        ta.coeff_rows = (int)p.Mpad;
        ta.skip = skip; ta.skip_ld = p.n_vt; ta.skip_rows = (int)(p.Mpad / 128);
        ta.dlogp = dlogp; ta.targets = targets; ta.filter_eps = eps;
        ta.kbits = kbits; ta.kbits_ld = p.kbits_ld;
        ta.cold_out = cold_out; ta.cold_out_ld = n_vb; ta.cold_out_rows = n_rb;
        if ((e = qh::launch_tc_fwd(th, tw_logit, ta, head->bits, true, p.grid, st)))
            return cuda_fail(e, "tc_coeff");
        if (dh) {
            qh::TcDhArgs da{};
            da.scales = sc; da.biases = bi; da.V = head->V; da.H = head->H;
            da.count = count; da.err = err; da.rows = rows; da.dlogp = dlogp; da.dh_acc = dhp;
            da.slice_stride = p.Mpad * head->H;
            da.v_begin = (int64_t)vt0 * tr;
            da.n_k = (vt1 - vt0) * tr / 64;
            da.ks = p.S;  // <= the K steps of every chunk (plan_bwd)
            da.accumulate = c > 0;
            da.skip = skip; da.skip_ld = p.n_vt; da.skip_rows = (int)(p.Mpad / 128);
            da.kbits = kbits; da.kbits_ld = p.kbits_ld;
            if ((e = qh::launch_tc_dh(tcoef, tw_dh, da, head->bits, p.grid, st)))
                return cuda_fail(e, "tc_dh");
        }
        if (dw) {
            qh::TcDwArgs wa{};
            wa.V = head->V; wa.H = head->H; wa.count = count; wa.err = err;
            wa.v_begin = (int64_t)vt0 * tr;
            wa.chunk_rows = (vt1 - vt0) * tr;
            wa.dmax = dmax; wa.offs = offs; wa.idx = idx; wa.g = g; wa.rows = rows;
            wa.h = hb; wa.dw = dw;
            if ((e = qh::launch_tc_dw(tcoef_t, thp, wa, p.grid, st)))
                return cuda_fail(e, "tc_dw");
        }
    }
    hook_after(st);
    if (dw && (e = qh::launch_dw_poison(err, dw, head->V * (int64_t)head->H, st)))
        return cuda_fail(e, "dw_poison");
    if (dh &&
        (e = qh::launch_bwd_finalize(wq, sbx, head->V, head->H, head->bits, head->softcap, hb,
                                     pos, targets, dlogp, dhp, p.S, p.Mpad, err, dh, M, st)))
        return cuda_fail(e, "bwd_finalize");
    return QHEAD_OK;
}

int qhead_bwd(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
              const uint8_t* mask, const float* lse, const float* dlogp, float* dh,
              void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(head, h, M, targets, mask, lse, dlogp, dh, nullptr, nullptr, 0.f, false,
                    nullptr, workspace,
                    workspace_bytes, stream);
}

int qhead_fwd(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
              const uint8_t* mask, float* logp, float* lse, int32_t* argmax, void* workspace,
              size_t workspace_bytes, void* stream) {
    return fwd_impl(head, h, M, targets, mask, logp, lse, argmax, nullptr, workspace,
                    workspace_bytes, stream);
}

int qhead_fwd_blockmax(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                       const uint8_t* mask, float* logp, float* lse, int32_t* argmax,
                       float* block_max, void* workspace, size_t workspace_bytes, void* stream) {
    HookScope hooks;
    if (!block_max && M > 0) {
        g_err.clear();
        return fail(QHEAD_EINVAL, "block_max is required");
    }
    return fwd_impl(head, h, M, targets, mask, logp, lse, argmax, block_max, workspace,
                    workspace_bytes, stream);
}

int qhead_bwd_dw(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                 const uint8_t* mask, const float* lse, const float* dlogp, float* dh, float* dw,
                 void* workspace, size_t workspace_bytes, void* stream) {
    HookScope hooks;
    if (!dw) {
        g_err.clear();
        return fail(QHEAD_EINVAL, "dw is required (qhead_bwd computes dh alone)");
    }
    return bwd_impl(head, h, M, targets, mask, lse, dlogp, dh, dw, nullptr, 0.f, false, nullptr,
                    workspace,
                    workspace_bytes, stream);
}

size_t qhead_bwd_blockskip_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    BwdPlan p;
    if (plan_bwd(head, M, &p, false, true)) return (size_t)-1;
    return p.total;
}

int qhead_bwd_blockskip(const qhead_head* head, const void* h, int64_t M,
                        const int32_t* targets, const uint8_t* mask, const float* lse,
                        const float* dlogp, const float* block_max, float eps, float* dh,
                        void* workspace, size_t workspace_bytes, void* stream) {
    HookScope hooks;
    if (M > 0 && !block_max) {
        g_err.clear();
        return fail(QHEAD_EINVAL, "block_max is required");
    }
    if (!(eps >= 0.f) || eps > 1.f) {
        g_err.clear();
        return fail(QHEAD_EINVAL, "eps must lie in [0, 1]");
    }
    return bwd_impl(head, h, M, targets, mask, lse, dlogp, dh, nullptr, block_max, eps, false,
                    nullptr, workspace,
                    workspace_bytes, stream);
}

size_t qhead_bwd_filter_workspace(const qhead_head* head, int64_t M) {
    g_err.clear();
    if (check_head(head)) return (size_t)-1;
    if (M < 0) { fail(QHEAD_EINVAL, "M < 0"); return (size_t)-1; }
    if (M == 0) return 0;
    BwdPlan p;
    if (plan_bwd(head, M, &p, false, false, true)) return (size_t)-1;
    return p.total;
}

int qhead_bwd_filter(const qhead_head* head, const void* h, int64_t M, const int32_t* targets,
                     const uint8_t* mask, const float* lse, const float* dlogp, float eps,
                     float* dh, uint8_t* cold, void* workspace, size_t workspace_bytes,
                     void* stream) {
    HookScope hooks;
    if (!(eps >= 0.f)) {
        g_err.clear();
        return fail(QHEAD_EINVAL, "eps must be >= 0");
    }
    return bwd_impl(head, h, M, targets, mask, lse, dlogp, dh, nullptr, nullptr, eps, true, cold,
                    workspace, workspace_bytes, stream);
}

int qhead_verify(const qhead_head* head, const void* h, int64_t B, int64_t W,
                 const int32_t* draft, const uint8_t* mask, float* lse, int32_t* argmax,
                 int32_t* n_accept, int32_t* next_token, void* workspace, size_t workspace_bytes,
                 void* stream) {
    HookScope hooks;
    g_err.clear();
    if (B < 0) return fail(QHEAD_EINVAL, "B < 0");
    if (W < 1 || W > (int64_t)1 << 20) return fail(QHEAD_EINVAL, "W must be in [1, 2^20]");
    if (B > 0 && B > (((int64_t)1 << 31) - qh::kRowPad) / W)
        return fail(QHEAD_EINVAL, "B * W too large");
    if (B == 0) return QHEAD_OK;
    if (!argmax || !n_accept) return fail(QHEAD_EINVAL, "argmax and n_accept are required");
    if (W > 1 && !draft) return fail(QHEAD_EINVAL, "draft is required when W > 1");
    const int rc = qhead_fwd(head, h, B * W, nullptr, mask, nullptr, lse, argmax, workspace,
                             workspace_bytes, stream);
    if (rc) return rc;
    cudaError_t e = qh::launch_accept_prefix(argmax, draft, B, (int)W, n_accept, next_token,
                                             static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "accept_prefix");
    return QHEAD_OK;
}

}  // extern "C"

namespace qh {

namespace {
std::mutex g_cache_mu;
std::map<std::pair<const void*, int>, int> g_smem_limit;  // (kernel, device) -> bytes allowed
std::map<int, int> g_sms;                                 // device -> SM count
}  // namespace

cudaError_t ensure_smem_limit(const void* func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    int& allowed = g_smem_limit[{func, dev}];
    if (allowed >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) allowed = bytes;
    return e;
}

cudaError_t launch_dependent(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             void** args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

int device_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
    return n;
}

}  // namespace qh
