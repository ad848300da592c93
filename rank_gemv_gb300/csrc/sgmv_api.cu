// sgmv_api.cu -- the C ABI declared in include/sgmv.h: argument checks,
// launch-shape choice and dispatch, host-side grouping, device error word.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "sgmv.h"
#include "sgmv_internal.h"
#include "sgmv_fused.h"
#include "sgmv_gather.h"

// Sticky device error word of this library (first reported status wins).
__device__ int g_sgmv_error;

namespace {

using namespace sgmv;

thread_local char g_last_error[256] = "";
thread_local int g_launches = 0;  // kernels launched by this thread's last call
thread_local int g_inject_timeout = 0;  // sgmv_debug_inject_wait_timeout

void note(const char *what, cudaError_t e) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, cudaGetErrorString(e));
}

int cuda_status(const char *what, int e) {
    if (e == (int)cudaSuccess) return SGMV_OK;
    note(what, (cudaError_t)e);
    return SGMV_ERR_CUDA;
}

// Device address of the error word of the current device, looked up once per
// device with that device current.
int *error_word() {
    static std::mutex mu;
    static int *cache[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_sgmv_error);
        if (e != cudaSuccess) {
            note("cudaGetSymbolAddress(error word)", e);
            return nullptr;
        }
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int round8(int64_t v) { return (int)((v + 7) / 8 * 8); }
int floor8(int64_t v) { return (int)(v / 8 * 8); }
int floor16(int64_t v) { return (int)(v / 16 * 16); }
int elem_size(int dt) { return dt == SGMV_F32 ? 4 : 2; }
int rmax_of(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : 128; }

int check_common(int32_t T, int32_t L, int32_t r, int32_t S, const int32_t *seg_ptr,
                 const int32_t *idx, const int32_t *seg_ptr_host, int in_dtype) {
    if (T < 0 || L < 1 || S < 0 || r < 1) return SGMV_ERR_INVALID_ARG;
    if (r > 128) return SGMV_ERR_UNSUPPORTED;
    if (in_dtype != SGMV_F16 && in_dtype != SGMV_BF16) return SGMV_ERR_INVALID_ARG;
    if (S > 0 && (!seg_ptr || !idx)) return SGMV_ERR_INVALID_ARG;
    if (seg_ptr_host) {
        for (int32_t s = 0; s <= S; ++s)
            if (seg_ptr_host[s] < 0 || seg_ptr_host[s] > T) return SGMV_ERR_BAD_SEGMENTS;
        for (int32_t s = 0; s < S; ++s)
            if (seg_ptr_host[s + 1] < seg_ptr_host[s]) return SGMV_ERR_BAD_SEGMENTS;
    }
    return SGMV_OK;
}

int check_dim(int32_t H) {
    if (H < 1) return SGMV_ERR_INVALID_ARG;
    if (H % 8 != 0) return SGMV_ERR_ALIGNMENT;
    return SGMV_OK;
}

// Longest segment (host copy known) or -1.
int32_t longest(const int32_t *sp, int32_t S) {
    if (!sp) return -1;
    int32_t m = 0;
    for (int32_t s = 0; s < S; ++s) m = std::max(m, sp[s + 1] - sp[s]);
    return m;
}

// Tile slots for segments of length in [min_len, max_len], `rows` rows per
// tile: exact from the host copy of seg_ptr, else a bound that holds for any
// segmentation of T positions into S segments.
int64_t tile_slots(int32_t T, int32_t S, const int32_t *sp, int rows, int min_len, int max_len) {
    if (sp) {
        int64_t n = 0;
        for (int32_t s = 0; s < S; ++s) {
            const int32_t len = sp[s + 1] - sp[s];
            if (len > 0 && len >= min_len && len <= max_len) n += ceil_div(len, rows);
        }
        return n;
    }
    // sum over segments of ceil(len / rows) <= (T + S (rows - 1)) / rows
    int64_t b = ((int64_t)T + (int64_t)S * (rows - 1)) / rows;
    // short segments only: at most ceil(max_len / rows) tiles each
    if (max_len < INT_MAX) b = std::min<int64_t>(b, (int64_t)S * ceil_div(max_len, rows));
    // long segments only: at most T / min_len of them, one partial tile each
    if (min_len > 1) b = std::min<int64_t>(b, (int64_t)T / rows + (int64_t)T / min_len);
    return b;
}

int cc_launch(int in_dtype, const CCLaunch &l) {
    return in_dtype == SGMV_F16 ? cc_launch_f16(l) : cc_launch_bf16(l);
}

// CTAs per cluster for the shrink side: largest of 8/4/2/1 that leaves every
// CTA at least 64 columns of H1 (and of H2 when it also expands).
int choose_cluster(int32_t H1, int32_t H2) {
    int cl = 8;
    while (cl > 1 && (H1 < cl * 64 || (H2 > 0 && H2 < cl * 64))) cl >>= 1;
    return cl;
}

// Streaming multiprocessors of the current device (looked up once per device).
int num_sms() {
    static std::mutex mu;
    static int cache[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// Encodes the B tensor map, then launches.  With H2 and every CTA's first
// column multiples of 256, B is viewed as [L][H2/256][r][256] so that one
// copy brings a whole chunk; otherwise as [L][r][H2], one copy per 256 columns.
int stream_launch(int in_dtype, StreamLaunch &l) {
    StreamParams &p = l.p;
    p.inject = g_inject_timeout;
    const bool bf16 = in_dtype == SGMV_BF16;
    const cuuint64_t es = 2;
    if (p.np < 1 || p.np > kStreamMaxProblems) return (int)cudaErrorInvalidValue;
    p.b4d = 0;
    if (p.H2 % 256 == 0 && p.jc % 256 == 0) {
        const cuuint64_t dims[4] = {256, (cuuint64_t)p.r, (cuuint64_t)p.H2 / 256, (cuuint64_t)p.L};
        const cuuint64_t strides[3] = {(cuuint64_t)p.H2 * es, 256 * es,
                                       (cuuint64_t)p.r * p.H2 * es};
        const cuuint32_t box[4] = {256, (cuuint32_t)p.r, (cuuint32_t)(p.hn / 256), 1};
        p.b4d = 1;
        for (int q = 0; q < p.np && p.b4d; ++q)
            p.b4d = tmap_encode(&p.tmap_b[q], bf16, 4, p.B[q], dims, strides, box, false) ? 1 : 0;
    }
    if (!p.b4d) {
        const cuuint64_t dims[3] = {(cuuint64_t)p.H2, (cuuint64_t)p.r, (cuuint64_t)p.L};
        const cuuint64_t strides[2] = {(cuuint64_t)p.H2 * es, (cuuint64_t)p.r * p.H2 * es};
        const cuuint32_t box[3] = {256, (cuuint32_t)p.r, 1};
        for (int q = 0; q < p.np; ++q)
            if (!tmap_encode(&p.tmap_b[q], bf16, 3, p.B[q], dims, strides, box, false))
                return (int)cudaErrorInvalidValue;
    }
    return in_dtype == SGMV_F16 ? stream_launch_f16(l) : stream_launch_bf16(l);
}

// Shared memory the streaming kernel may use for its ring and buffers.
// Two CTAs fit on one SM (228 KB), so the next call's CTAs can start, group
// and request their weights while this call's CTAs still run.  A CTA that
// takes a whole SM keeps its ring to 170 KB: on the Llama-2-7B stack (stages
// of 34 KB) four stages measured 0.708 of the HBM peak against 0.698 for
// five and 0.692 for three, and a single q projection 0.574 against 0.550 for
// five; more bytes in flight per SM only lengthen the copies' latency.
constexpr uint32_t kStreamSmemBudget = 110u * 1024u;
constexpr uint32_t kStreamSmemMax = 170u * 1024u;

}  // namespace

void sgmv::note_cuda_error(const char *what, cudaError_t e) { note(what, e); }

int *sgmv::device_error_word() { return error_word(); }

// Launch shape of the streaming kernel for a batch of T rows in S segments
// (the last max_len rows long at most), or false when the kernel does not
// apply (r not a multiple of 4 or above 64, or more tiles per cluster than its
// table holds).  Rows per tile: 1 when segments average up to 2 rows (every
// row streams its adapter on its own; rows that share an adapter read it
// again from L2), up to 8 for longer segments, whose rows then share each
// staged weight chunk.  The cluster size -- and with it the summation order
// -- depends on T and the dimensions only, never on the segmentation: as
// many CTAs per tile (8, 4, 2, 1) as keep CTAs x T within the SM count (within
// twice the SM count, at two CTAs per SM, for 39..64 rows), each with at least
// 64 columns of H1 and of H2.
bool sgmv::stream_shape(int32_t T, int32_t S, const int32_t *seg_ptr_host, int32_t max_len,
                        int32_t H1, int32_t H2, int32_t r, int in_dtype, int y_dtype,
                        StreamLaunch &l, bool grouped, int np) {
    if (r % 4 != 0 || r > 64 || T <= 0 || S <= 0) return false;
    if (np < 1 || np > kStreamMaxProblems || (grouped && np != 1)) return false;
    const int64_t avg = ceil_div(T, S);
    // The one-launch grouped form cannot see the segments.  Above 32 rows
    // tiles of two rows halve the streaming of repeated adapters (measured on
    // a Zipf batch of 64 rows in clusters of four at two CTAs per SM, us per
    // call back to back: 7.46 with two-row tiles, 8.03 with one, 9.21 with
    // four, 12.55 with eight: taller tiles leave a few CTAs compute-bound).
    // Up to 32 rows, one-row tiles measured faster (one shared adapter, 32
    // rows: 4.0 against 4.4 us).  Tile height does not change any row's
    // summation order.
    const int trows = grouped && T > 32 ? 2 : avg <= 2 ? 1 : avg <= 4 ? 2 : avg <= 8 ? 4 : 8;
    // units: (problem, tile) pairs
    const int64_t slots = tile_slots(T, S, seg_ptr_host, trows, 1, max_len) * np;
    if (slots <= 0) return false;
    const int nsm = num_sms();
    if (nsm <= 0) return false;
    int cl = 8;
    while (cl > 1 && ((int64_t)cl * T > nsm || H1 < cl * 64 || H2 < cl * 64)) cl >>= 1;
    // 39..64 rows: clusters twice as large at two CTAs per SM, each CTA
    // streaming half as much of its tile's adapter (measured on a Zipf batch
    // of 64 rows: 7.50 against 8.85 us back to back, 14.96 against 17.04
    // isolated).  Like the rule above, a function of T and the dimensions.
    bool half = false;
    if (np == 1 && 4 * (int64_t)T > nsm && T <= kGroupMaxT && cl < 8 && H1 >= 2 * cl * 64 &&
        H2 >= 2 * cl * 64) {
        cl *= 2;
        half = true;
    }
    // several problems: single-CTA clusters only (large batches), where the
    // kernel has an instantiation for them
    if (np > 1 && cl != 1) return false;
    const int64_t gmax = std::max<int64_t>(1, (half ? 2 : 1) * (int64_t)nsm / cl);
    if (ceil_div((int64_t)T * np, gmax) > kStreamMaxTiles) return false;
    StreamParams &p = l.p;
    const int rk = r <= 16 ? 16 : r <= 32 ? 32 : 64;
    p.np = np;
    p.cl = cl;
    p.G = (int32_t)std::min<int64_t>(slots, gmax);
    // A cluster of several CTAs gets one tile (cl * T <= #SMs above makes
    // G = slots); only single-CTA clusters walk several tiles.  Clusters that
    // walked several tiles each (eight CTAs, seven tiles, forced for a
    // measurement) faulted the GPU once, cause not found: never launched.
    if (cl > 1 && p.G < slots) return false;
    p.hc = round8(ceil_div(H1, cl));
    p.jc = round8(ceil_div(H2, cl));
    if (H2 % 256 == 0) {  // lets B chunks start on 256-column blocks (one copy each)
        const int32_t jc256 = (int32_t)(ceil_div(H2, 256LL * cl) * 256);
        if ((int64_t)(cl - 1) * jc256 < H2) p.jc = jc256;
    }
    p.hn = kStreamChunkElems / rk;
    const uint32_t es = (uint32_t)elem_size(in_dtype), ys = (uint32_t)elem_size(y_dtype);
    const uint32_t w = align_up((uint32_t)(p.hn * r) * es, 128);
    const uint32_t act = align_up((uint32_t)trows * (uint32_t)p.hn * std::max(es, ys), 128);
    p.stage_bytes = w + act;
    p.act_off = w;
    // 16 compute warps when a CTA owns whole tiles (more warps to hide the
    // compute warps' latencies; one CTA per SM anyway); a function of T and
    // the dimensions only, like the cluster size: it fixes the summation order
    l.cw = cl == 1 ? 16 : 8;
    const uint32_t red = (uint32_t)l.cw * 8u * (uint32_t)rk * 4u;
    const uint32_t recv = cl > 1 ? 2u * (uint32_t)cl * 8u * (uint32_t)rk * 4u : 0u;
    const uint32_t vbytes = 2u * 8u * (uint32_t)rk * 4u;
    const uint32_t tab = (uint32_t)kStreamMaxTiles * 12u * 4u;
    const int64_t chunks = ceil_div(slots, p.G) * (ceil_div(p.hc, p.hn) + ceil_div(p.jc, p.hn));
    const uint32_t fixed = red + recv + vbytes + tab;
    // A CTA with few chunks to stream (small batches) keeps to half an SM, so
    // the next call's CTAs can start beside it and request their weights
    // early.  A CTA with many chunks, or with large stages, takes a whole SM
    // for a deeper ring: more bytes in flight per SM.
    int64_t nst = (int64_t)(kStreamSmemBudget - fixed) / p.stage_bytes;
    if (!half && (nst < 3 || chunks > 2 * nst))
        nst = (int64_t)(kStreamSmemMax - fixed) / p.stage_bytes;
    if (half && nst < 2) return false;  // two CTAs per SM need two stages each (r <= 64 has them)
    nst = std::min<int64_t>(std::min<int64_t>(nst, kStreamMaxStages), chunks);
    if (nst < 1) return false;
    p.nst = (int32_t)nst;
    p.trows = trows;
    p.red_off = (uint32_t)nst * p.stage_bytes;
    p.recv_off = p.red_off + red;
    p.v_off = p.recv_off + recv;
    p.tab_off = p.v_off + vbytes;
    p.smem_bytes = p.tab_off + tab;
    l.rk = rk;
    l.in_dtype = in_dtype;
    l.y_dtype = y_dtype;
    return true;
}

namespace {

void stage_sizes(CCParams &p, int mode, int elem);

// Fill the derived launch parameters once rows, r, cl, hc and jc are set.
void finish(CCParams &p, int mode, int in_dtype, int y_dtype) {
    p.rmax = rmax_of(p.r);
    p.ysize = elem_size(y_dtype);
    stage_sizes(p, mode, elem_size(in_dtype));
    // prefetch y rows when the CTA's whole H2 slice is staged as one chunk
    p.y_pref = (mode != kShrink && p.jc <= p.js) ? 1 : 0;
}

void stage_sizes(CCParams &p, int mode, int elem) {
    if (mode != kExpand) {
        // Sized for kRowsMax rows whatever the tile height, so the chunking of
        // H1 (and with it the summation order of every row's v) does not
        // depend on how segments are cut into tiles.
        p.hs = std::min(p.hc, floor16(kStageBytes / ((int64_t)(p.r + kRowsMax) * elem)));
        p.ax_stages = ceil_div(p.hc, p.hs) > 1 ? 2 : 1;
    } else {
        p.hs = 8;
        p.ax_stages = 1;
    }
    if (mode != kShrink) {
        p.js = std::min(p.jc, floor8(kStageBytes / ((int64_t)p.r * elem)));
        p.b_stages = ceil_div(p.jc, p.js) > 1 ? 2 : 1;
    } else {
        p.js = 8;
        p.b_stages = 1;
    }
}

}  // namespace

extern "C" {

const char *sgmv_status_string(int status) {
    switch (status) {
        case SGMV_OK: return "SGMV_OK";
        case SGMV_ERR_INVALID_ARG: return "SGMV_ERR_INVALID_ARG";
        case SGMV_ERR_UNSUPPORTED: return "SGMV_ERR_UNSUPPORTED";
        case SGMV_ERR_ALIGNMENT: return "SGMV_ERR_ALIGNMENT";
        case SGMV_ERR_BAD_INDEX: return "SGMV_ERR_BAD_INDEX";
        case SGMV_ERR_CUDA: return "SGMV_ERR_CUDA";
        case SGMV_ERR_WORKSPACE: return "SGMV_ERR_WORKSPACE";
        case SGMV_ERR_TIMEOUT: return "SGMV_ERR_TIMEOUT";
        case SGMV_ERR_BAD_SEGMENTS: return "SGMV_ERR_BAD_SEGMENTS";
        default: return "SGMV_ERR_UNKNOWN";
    }
}

const char *sgmv_last_error_string(void) { return g_last_error; }

int sgmv_last_launch_count(void) { return g_launches; }

int32_t sgmv_max_segments(int32_t T, int32_t L) {
    if (T <= 0 || L < 0) return 0;
    return (int32_t)std::min<int64_t>(T, (int64_t)L + 1);
}

int sgmv_build_segments(const int32_t *row_adapter, int32_t T, int32_t L, int32_t *perm,
                        int32_t *seg_ptr, int32_t *idx, int32_t *S) {
    if (T < 0 || L < 1 || !seg_ptr || !S) return SGMV_ERR_INVALID_ARG;
    if (T > 0 && (!row_adapter || !perm || !idx)) return SGMV_ERR_INVALID_ARG;
    for (int32_t t = 0; t < T; ++t)
        if (row_adapter[t] < -1 || row_adapter[t] >= L) return SGMV_ERR_BAD_INDEX;
    // Counting sort on key = id + 1: counts, then start positions.
    std::vector<int32_t> start((size_t)L + 1, 0);
    for (int32_t t = 0; t < T; ++t) ++start[(size_t)row_adapter[t] + 1];
    int32_t pos = 0, s = 0;
    for (int32_t b = 0; b <= L; ++b) {
        const int32_t c = start[b];
        if (c > 0) {
            seg_ptr[s] = pos;
            idx[s] = b - 1;
            ++s;
        }
        start[b] = pos;
        pos += c;
    }
    seg_ptr[s] = T;
    for (int32_t t = 0; t < T; ++t) perm[start[(size_t)row_adapter[t] + 1]++] = t;
    *S = s;
    return SGMV_OK;
}

int sgmv_build_segments_device(const int32_t *row_adapter, int32_t T, int32_t L, int32_t *perm,
                               int32_t *seg_ptr, int32_t *idx, int32_t *S, void *stream) {
    g_launches = 0;
    if (T < 0 || L < 1 || !seg_ptr || !S) return SGMV_ERR_INVALID_ARG;
    if (T > 0 && (!row_adapter || !perm || !idx)) return SGMV_ERR_INVALID_ARG;
    if (L > 32767) return SGMV_ERR_UNSUPPORTED;
    int *err = error_word();
    if (!err) return SGMV_ERR_CUDA;
    const int st = cuda_status("build_segments kernel",
                               build_segments_launch(row_adapter, T, L, perm, seg_ptr, idx, S,
                                                     sgmv_max_segments(T, L), err,
                                                     static_cast<cudaStream_t>(stream)));
    if (st == SGMV_OK) g_launches = 1;
    return st;
}

size_t sgmv_workspace_bytes(int32_t T, int32_t H1, int32_t H2, int32_t r) {
    (void)H1;
    (void)H2;
    if (T <= 0 || r <= 0) return 0;
    // v as two 16-bit halves, [T][r] each, 256-byte aligned, then 256 bytes
    // for the tensor-core expand's claim counter
    const size_t half = ((size_t)T * (size_t)r * 2u + 255u) / 256u * 256u;
    return 2u * half + 256u;
}

int sgmv_shrink(float *v, const void *x, const void *A, int in_dtype, const int32_t *perm,
                const int32_t *seg_ptr, const int32_t *idx, int32_t S, const int32_t *seg_ptr_host,
                int32_t T, int32_t L, int32_t H1, int32_t r, void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, S, seg_ptr, idx, seg_ptr_host, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if (T == 0 || S == 0) return SGMV_OK;
    if (!v || !x || !A) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(x) || !aligned16(A)) return SGMV_ERR_ALIGNMENT;

    CCLaunch l = {};
    CCParams &p = l.p;
    p.x = x;
    p.A = A;
    p.v_out = v;
    p.perm = perm;
    p.seg_ptr = seg_ptr;
    p.idx = idx;
    p.S = S;
    p.T = T;
    p.L = L;
    p.H1 = H1;
    p.H2 = 8;
    p.r = r;
    const int32_t mx = longest(seg_ptr_host, S);
    p.rows = mx > 0 ? std::min(kRowsMax, mx) : kRowsMax;
    p.min_len = 1;
    p.max_len = INT_MAX;
    p.scale = 0.f;
    // CTAs per tile: as many as keep T x CL (the grid when every row is its
    // own segment) within two CTAs per SM, so that short segments do not
    // multiply into several waves of small CTAs (at T = 128 on 128 adapters,
    // 1,024 CTAs of 16 KB each; clusters of 2 measured 9% faster in the fused
    // layer).  A function of T and H1 only, like the summation order it fixes.
    int cl = choose_cluster(H1, 0);
    const int nsm = num_sms();
    while (cl > 1 && nsm > 0 && (int64_t)T * cl > 2 * (int64_t)nsm) cl >>= 1;
    p.hc = round8(ceil_div(H1, cl));
    p.jc = 8;
    p.cl = cl;
    finish(p, kShrink, in_dtype, SGMV_F32);
    const int64_t slots = tile_slots(T, S, seg_ptr_host, p.rows, 1, INT_MAX);
    if (slots == 0) return SGMV_OK;
    if (slots > 65535) return SGMV_ERR_UNSUPPORTED;
    if (!(p.err = error_word())) return SGMV_ERR_CUDA;
    l.mode = kShrink;
    l.y_dtype = SGMV_F32;
    l.rmax = rmax_of(r);
    l.grid = dim3((unsigned)cl, (unsigned)slots, 1);
    l.cluster = cl;
    l.stream = static_cast<cudaStream_t>(stream);
    l.pdl = true;
    st = cuda_status("shrink kernel", cc_launch(in_dtype, l));
    if (st == SGMV_OK) g_launches = 1;
    return st;
}

int sgmv_expand(void *y, int y_dtype, const float *v, const void *B, int in_dtype, float scale,
                const int32_t *perm, const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H2, int32_t r,
                void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, S, seg_ptr, idx, seg_ptr_host, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    if (T == 0 || S == 0) return SGMV_OK;
    if (!y || !v || !B) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(v) || !aligned16(B)) return SGMV_ERR_ALIGNMENT;

    CCLaunch l = {};
    CCParams &p = l.p;
    p.y = y;
    p.B = B;
    p.v_in = v;
    p.perm = perm;
    p.seg_ptr = seg_ptr;
    p.idx = idx;
    p.S = S;
    p.T = T;
    p.L = L;
    p.H1 = 8;
    p.H2 = H2;
    p.r = r;
    const int32_t mx = longest(seg_ptr_host, S);
    p.rows = mx > 0 ? std::min(kRowsMax, mx) : kRowsMax;
    p.min_len = 1;
    p.max_len = INT_MAX;
    p.scale = scale;
    const int nx = (int)std::max<int64_t>(1, ceil_div(H2, 512));
    p.jc = round8(ceil_div(H2, nx));
    p.hc = 8;
    p.cl = 1;
    finish(p, kExpand, in_dtype, y_dtype);
    const int64_t slots = tile_slots(T, S, seg_ptr_host, p.rows, 1, INT_MAX);
    if (slots == 0) return SGMV_OK;
    if (slots > 65535) return SGMV_ERR_UNSUPPORTED;
    if (!(p.err = error_word())) return SGMV_ERR_CUDA;
    l.mode = kExpand;
    l.y_dtype = y_dtype;
    l.rmax = rmax_of(r);
    l.grid = dim3((unsigned)ceil_div(H2, p.jc), (unsigned)slots, 1);
    l.cluster = 1;
    l.stream = static_cast<cudaStream_t>(stream);
    l.pdl = true;
    st = cuda_status("expand kernel", cc_launch(in_dtype, l));
    if (st == SGMV_OK) g_launches = 1;
    return st;
}

int sgmv_apply(void *y, int y_dtype, const void *x, const void *A, const void *B, int in_dtype,
               float scale, const int32_t *perm, const int32_t *seg_ptr, const int32_t *idx,
               int32_t S, const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H1,
               int32_t H2, int32_t r, void *workspace, size_t workspace_bytes, void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, S, seg_ptr, idx, seg_ptr_host, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    if (workspace && workspace_bytes < sgmv_workspace_bytes(T, H1, H2, r)) return SGMV_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return SGMV_ERR_ALIGNMENT;
    if (T == 0 || S == 0) return SGMV_OK;
    if (!y || !x || !A || !B) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(x) || !aligned16(A) || !aligned16(B))
        return SGMV_ERR_ALIGNMENT;

    int *err = error_word();
    if (!err) return SGMV_ERR_CUDA;
    // Dispatch, when a workspace holds v and r suits the tensor-core tiles:
    // in prefill-like batches (segments average 8 rows or more) every segment
    // goes to the tensor cores, which read each segment's weights once as the
    // CUDA-core kernel would, and no CUDA-core launch is made; otherwise
    // segments of at least kTcMinLen rows go to the tensor cores and the rest
    // to the CUDA-core kernel.  The choice depends on T and S only, so host
    // and device metadata give the same bits.
    bool use_tc = workspace != nullptr && (r == 64 || r == 128) && T >= kTcMinLen;
    int64_t tc_slots = 0;
    int32_t tc_min = kTcMinLen;
    if (use_tc) {
        if ((int64_t)T >= 8LL * S) tc_min = 1;
        tc_slots = tile_slots(T, S, seg_ptr_host, 128, tc_min, INT_MAX);
        if (tc_slots > 65535) return SGMV_ERR_UNSUPPORTED;
        use_tc = tc_slots > 0;
    }
    const int32_t cc_max_len = use_tc ? tc_min - 1 : INT_MAX;

    CCLaunch l = {};
    CCParams &p = l.p;
    p.y = y;
    p.x = x;
    p.A = A;
    p.B = B;
    p.perm = perm;
    p.seg_ptr = seg_ptr;
    p.idx = idx;
    p.S = S;
    p.T = T;
    p.L = L;
    p.H1 = H1;
    p.H2 = H2;
    p.r = r;
    const int32_t mx = longest(seg_ptr_host, S);
    p.rows = mx > 0 ? std::min(kRowsMax, mx) : kRowsMax;
    p.min_len = 1;
    p.max_len = cc_max_len;
    p.scale = scale;
    const int cl = choose_cluster(H1, H2);
    p.hc = round8(ceil_div(H1, cl));
    p.jc = round8(ceil_div(H2, cl));
    p.cl = cl;
    finish(p, kFused, in_dtype, y_dtype);
    const int64_t slots = tile_slots(T, S, seg_ptr_host, p.rows, 1, cc_max_len);
    if (slots > 65535) return SGMV_ERR_UNSUPPORTED;
    p.err = err;
    StreamLaunch sl = {};
    if (slots > 0 &&
        stream_shape(T, S, seg_ptr_host, cc_max_len, H1, H2, r, in_dtype, y_dtype, sl, false)) {
        StreamParams &q = sl.p;
        q.np = 1;
        q.y[0] = y;
        q.x[0] = x;
        q.A[0] = A;
        q.B[0] = B;
        q.perm = perm;
        q.seg_ptr = seg_ptr;
        q.idx = idx;
        q.err = err;
        q.S = S;
        q.T = T;
        q.L = L;
        q.H1 = H1;
        q.H2 = H2;
        q.r = r;
        q.min_len = 1;
        q.max_len = cc_max_len;
        q.scale = scale;
        sl.grouped = false;
        sl.stream = static_cast<cudaStream_t>(stream);
        st = cuda_status("streaming kernel", stream_launch(in_dtype, sl));
        if (st != SGMV_OK) return st;
        g_launches = 1;
    } else if (slots > 0) {
        l.mode = kFused;
        l.y_dtype = y_dtype;
        l.rmax = rmax_of(r);
        l.grid = dim3((unsigned)cl, (unsigned)slots, 1);
        l.cluster = cl;
        l.stream = static_cast<cudaStream_t>(stream);
        l.pdl = true;
        st = cuda_status("fused kernel", cc_launch(in_dtype, l));
        if (st != SGMV_OK) return st;
        g_launches = 1;
    }
    if (!use_tc) return SGMV_OK;

    TCArgs g = {};
    g.y = y;
    g.x = x;
    g.A = A;
    g.B = B;
    g.perm = perm;
    g.seg_ptr = seg_ptr;
    g.idx = idx;
    g.err = err;
    const size_t half = ((size_t)T * (size_t)r * 2u + 255u) / 256u * 256u;
    g.vhi = workspace;
    g.vlo = static_cast<uint8_t *>(workspace) + half;
    g.S = S;
    g.T = T;
    g.L = L;
    g.H1 = H1;
    g.H2 = H2;
    g.r = r;
    g.min_len = tc_min;
    g.max_len = INT_MAX;
    g.scale = scale;
    g.in_dtype = in_dtype;
    g.y_dtype = y_dtype;
    g.slots = tc_slots;
    g.nsm = num_sms();
    g.stream = static_cast<cudaStream_t>(stream);
    st = cuda_status("tensor-core kernels", tc_launch(g));
    if (st == SGMV_OK) g_launches += 2;
    return st;
}

int sgmv_apply_multi(int32_t P, void *const *y, int y_dtype, const void *const *x,
                     const void *const *A, const void *const *B, int in_dtype, float scale,
                     const int32_t *perm, const int32_t *seg_ptr, const int32_t *idx, int32_t S,
                     const int32_t *seg_ptr_host, int32_t T, int32_t L, int32_t H1, int32_t H2,
                     int32_t r, void *stream) {
    g_launches = 0;
    if (P < 1 || P > kStreamMaxProblems || !y || !x || !A || !B) return SGMV_ERR_INVALID_ARG;
    int st = check_common(T, L, r, S, seg_ptr, idx, seg_ptr_host, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    if (T == 0 || S == 0) return SGMV_OK;
    for (int q = 0; q < P; ++q) {
        if (!y[q] || !x[q] || !A[q] || !B[q]) return SGMV_ERR_INVALID_ARG;
        if (!aligned16(y[q]) || !aligned16(x[q]) || !aligned16(A[q]) || !aligned16(B[q]))
            return SGMV_ERR_ALIGNMENT;
    }
    int *err = error_word();
    if (!err) return SGMV_ERR_CUDA;
    // One launch of the streaming kernel's multi-problem instantiation for all
    // P problems (P = 1 too: a serving loop whose calls all come here then
    // runs one kernel; alternating it with the single-problem kernel made a
    // Llama-2-7B step 14 % slower, 2.456 against 2.150 ms) when its launch
    // shape allows: one-CTA clusters, as P separate calls would have them
    // (the same bits); otherwise P separate calls.
    StreamLaunch sl = {};
    if (stream_shape(T, S, seg_ptr_host, INT_MAX, H1, H2, r, in_dtype, y_dtype, sl, false, P) &&
        sl.p.cl == 1) {
        sl.multi = true;
        StreamParams &q = sl.p;
        for (int k = 0; k < P; ++k) {
            q.y[k] = y[k];
            q.x[k] = x[k];
            q.A[k] = A[k];
            q.B[k] = B[k];
        }
        q.perm = perm;
        q.seg_ptr = seg_ptr;
        q.idx = idx;
        q.err = err;
        q.S = S;
        q.T = T;
        q.L = L;
        q.H1 = H1;
        q.H2 = H2;
        q.r = r;
        q.min_len = 1;
        q.max_len = INT_MAX;
        q.scale = scale;
        sl.grouped = false;
        sl.stream = static_cast<cudaStream_t>(stream);
        st = cuda_status("streaming kernel", stream_launch(in_dtype, sl));
        if (st == SGMV_OK) g_launches = 1;
        return st;
    }
    int launches = 0;
    for (int k = 0; k < P; ++k) {
        st = sgmv_apply(y[k], y_dtype, x[k], A[k], B[k], in_dtype, scale, perm, seg_ptr, idx, S,
                        seg_ptr_host, T, L, H1, H2, r, nullptr, 0, stream);
        launches += g_launches;
        if (st != SGMV_OK) break;
    }
    g_launches = launches;
    return st;
}

int sgmv_apply_rows(void *y, int y_dtype, const void *x, const void *A, const void *B,
                    int in_dtype, float scale, const int32_t *row_adapter, int32_t T, int32_t L,
                    int32_t H1, int32_t H2, int32_t r, int32_t *perm, int32_t *seg_ptr,
                    int32_t *idx, int32_t *S, void *workspace, size_t workspace_bytes,
                    void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, 0, nullptr, nullptr, nullptr, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    const bool meta = perm != nullptr;
    if (meta != (seg_ptr != nullptr) || meta != (idx != nullptr) || meta != (S != nullptr))
        return SGMV_ERR_INVALID_ARG;
    if (workspace && workspace_bytes < sgmv_workspace_bytes(T, H1, H2, r)) return SGMV_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return SGMV_ERR_ALIGNMENT;
    if (T == 0)
        return meta ? sgmv_build_segments_device(row_adapter, T, L, perm, seg_ptr, idx, S, stream)
                    : SGMV_OK;
    if (!row_adapter || !y || !x || !A || !B) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(x) || !aligned16(A) || !aligned16(B))
        return SGMV_ERR_ALIGNMENT;
    const int32_t smax = sgmv_max_segments(T, L);
    // T <= kGroupMaxT < kTcMinLen: no segment can reach the tensor cores
    if (T <= kGroupMaxT) {
        // One launch: every CTA groups the rows itself.
        int *err = error_word();
        if (!err) return SGMV_ERR_CUDA;
        StreamLaunch sl = {};
        if (stream_shape(T, smax, nullptr, INT_MAX, H1, H2, r, in_dtype, y_dtype, sl, true)) {
            StreamParams &q = sl.p;
            q.np = 1;
            q.y[0] = y;
            q.x[0] = x;
            q.A[0] = A;
            q.B[0] = B;
            q.err = err;
            q.row_adapter = row_adapter;
            q.perm_out = perm;
            q.seg_out = seg_ptr;
            q.idx_out = idx;
            q.S_out = S;
            q.S_max = smax;
            q.T = T;
            q.L = L;
            q.H1 = H1;
            q.H2 = H2;
            q.r = r;
            q.min_len = 1;
            q.max_len = INT_MAX;
            q.scale = scale;
            sl.grouped = true;
            sl.stream = static_cast<cudaStream_t>(stream);
            st = cuda_status("grouped streaming kernel", stream_launch(in_dtype, sl));
            if (st == SGMV_OK) g_launches = 1;
            return st;
        }
        CCLaunch l = {};
        CCParams &p = l.p;
        p.y = y;
        p.x = x;
        p.A = A;
        p.B = B;
        p.err = err;
        p.row_adapter = row_adapter;
        p.perm_out = perm;
        p.seg_out = seg_ptr;
        p.idx_out = idx;
        p.S_out = S;
        p.S_max = smax;
        p.S = 0;
        p.T = T;
        p.L = L;
        p.H1 = H1;
        p.H2 = H2;
        p.r = r;
        p.rows = kRowsMax;
        p.min_len = 1;
        p.max_len = INT_MAX;
        p.scale = scale;
        const int cl = choose_cluster(H1, H2);
        p.hc = round8(ceil_div(H1, cl));
        p.jc = round8(ceil_div(H2, cl));
        p.cl = cl;
        finish(p, kFused, in_dtype, y_dtype);
        const int64_t slots = ((int64_t)T + (int64_t)smax * (kRowsMax - 1)) / kRowsMax;
        l.mode = kGrouped;
        l.y_dtype = y_dtype;
        l.rmax = rmax_of(r);
        l.grid = dim3((unsigned)cl, (unsigned)slots, 1);
        l.cluster = cl;
        l.stream = static_cast<cudaStream_t>(stream);
        l.pdl = true;
        st = cuda_status("grouped fused kernel", cc_launch(in_dtype, l));
        if (st == SGMV_OK) g_launches = 1;
        return st;
    }
    // Larger batches, or long segments for the tensor cores: group into the
    // caller's metadata arrays, then the general update.
    if (!meta) return SGMV_ERR_INVALID_ARG;
    st = sgmv_build_segments_device(row_adapter, T, L, perm, seg_ptr, idx, S, stream);
    if (st != SGMV_OK) return st;
    st = sgmv_apply(y, y_dtype, x, A, B, in_dtype, scale, perm, seg_ptr, idx, smax, nullptr, T, L,
                    H1, H2, r, workspace, workspace_bytes, stream);
    g_launches += 1;
    return st;
}

int sgmv_load_adapter(void *A_pool, void *B_pool, int in_dtype, int32_t slot, const void *A_src,
                      const void *B_src, int32_t L, int32_t H1, int32_t H2, int32_t r,
                      void *stream) {
    g_launches = 0;
    if (!A_pool || !B_pool || !A_src || !B_src) return SGMV_ERR_INVALID_ARG;
    if (L < 1 || H1 < 1 || H2 < 1 || r < 1 || slot < 0 || slot >= L) return SGMV_ERR_INVALID_ARG;
    if (in_dtype != SGMV_F16 && in_dtype != SGMV_BF16) return SGMV_ERR_INVALID_ARG;
    const size_t a_bytes = (size_t)H1 * (size_t)r * 2u, b_bytes = (size_t)r * (size_t)H2 * 2u;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = cuda_status("adapter A copy",
                         cudaMemcpyAsync(static_cast<uint8_t *>(A_pool) + (size_t)slot * a_bytes,
                                         A_src, a_bytes, cudaMemcpyDefault, s));
    if (st != SGMV_OK) return st;
    return cuda_status("adapter B copy",
                       cudaMemcpyAsync(static_cast<uint8_t *>(B_pool) + (size_t)slot * b_bytes,
                                       B_src, b_bytes, cudaMemcpyDefault, s));
}

// Address under which the current device `dev` reads p, or null if it cannot
// read it directly: device memory of `dev`, or page-locked host memory mapped
// into the device's address space.  Pageable and other devices' memory give
// null (those copies go through the copy engine).
static const void *device_view(const void *p, int dev) {
    cudaPointerAttributes a = {};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // an unknown pointer: not an error of this call
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == dev ? p : nullptr;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

int sgmv_copy_gather(int32_t n, void *const *dst, const void *const *src, const uint64_t *bytes,
                     int32_t max_ctas, void *stream) {
    g_launches = 0;
    if (n < 0 || n > kGatherMaxCopies || max_ctas < 0) return SGMV_ERR_INVALID_ARG;
    if (n == 0) return SGMV_OK;
    if (!dst || !src || !bytes) return SGMV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (bytes[i] && (!dst[i] || !src[i])) return SGMV_ERR_INVALID_ARG;
    int dev = 0;
    int st = cuda_status("current device", cudaGetDevice(&dev));
    if (st != SGMV_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::vector<void *> kd;
    std::vector<const void *> ks;
    std::vector<uint64_t> kb;
    for (int i = 0; i < n; ++i) {
        if (!bytes[i]) continue;
        const void *sv = nullptr;
        void *dv = nullptr;
        if (bytes[i] % 16u == 0 && aligned16(src[i]) && aligned16(dst[i])) {
            sv = device_view(src[i], dev);
            dv = const_cast<void *>(device_view(dst[i], dev));
        }
        if (sv && dv && aligned16(sv) && aligned16(dv)) {
            kd.push_back(dv);
            ks.push_back(sv);
            kb.push_back(bytes[i]);
        } else {
            st = cuda_status("gather fallback copy",
                             cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyDefault, s));
            if (st != SGMV_OK) return st;
        }
    }
    if (kd.empty()) return SGMV_OK;
    const int cap = max_ctas > 0 ? max_ctas : 4 * std::max(1, num_sms());
    st = cuda_status("gather kernel",
                     gather_launch((int32_t)kd.size(), kd.data(), ks.data(), kb.data(), cap, s));
    if (st == SGMV_OK) g_launches = 1;
    return st;
}

// Workspace of the fused layer: v [T][r] fp32, the pair table and the v tiles,
// then the fp32 partials of split tiles; each part 256-byte aligned.
size_t fused_v_bytes(int32_t T, int32_t r) { return ((size_t)T * (size_t)r * 4u + 255u) / 256u * 256u; }

size_t sgmv_fused_workspace_bytes(int32_t T, int32_t H2, int32_t r) {
    if (T <= 0 || H2 <= 0 || r <= 0) return 0;
    return fused_v_bytes(T, r) + fused_prep_bytes(T, r) + fused_part_bytes(T, H2);
}

int sgmv_fused_linear_lora(void *y, int y_dtype, const void *x, const void *W, const void *A,
                           const void *B, int in_dtype, float scale, const int32_t *perm,
                           const int32_t *seg_ptr, const int32_t *idx, int32_t S, int32_t T,
                           int32_t L, int32_t H1, int32_t H2, int32_t r, void *workspace,
                           size_t workspace_bytes, void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, S, seg_ptr, idx, nullptr, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    if (T > kFusedMaxT || r > kFusedMaxR) return SGMV_ERR_UNSUPPORTED;
    if (T == 0) return SGMV_OK;
    if (!y || !x || !W || !A || !B) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(x) || !aligned16(W) || !aligned16(A) || !aligned16(B))
        return SGMV_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < sgmv_fused_workspace_bytes(T, H2, r))
        return SGMV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return SGMV_ERR_ALIGNMENT;
    int *err = error_word();
    if (!err) return SGMV_ERR_CUDA;
    int launches = 0;
    if (S > 0) {
        // v = x . A[idx] by sorted position, fp32, into the workspace
        st = sgmv_shrink(static_cast<float *>(workspace), x, A, in_dtype, perm, seg_ptr, idx, S,
                         nullptr, T, L, H1, r, stream);
        if (st != SGMV_OK) return st;
        launches = g_launches;
    }
    FusedArgs g = {};
    g.y = y;
    g.x = x;
    g.W = W;
    g.B = B;
    g.v = S > 0 ? static_cast<const float *>(workspace) : nullptr;
    g.perm = perm;
    g.seg_ptr = seg_ptr;
    g.idx = idx;
    g.err = err;
    g.S = S;
    g.T = T;
    g.L = L;
    g.H1 = H1;
    g.H2 = H2;
    g.r = r;
    g.scale = scale;
    g.in_dtype = in_dtype;
    g.y_dtype = y_dtype;
    g.prep = S > 0 ? static_cast<uint8_t *>(workspace) + fused_v_bytes(T, r) : nullptr;
    g.part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + fused_v_bytes(T, r) +
                                       fused_prep_bytes(T, r));
    g.nsm = num_sms();
    g.x_early = launches > 0;
    g.stream = static_cast<cudaStream_t>(stream);
    st = cuda_status("fused linear + LoRA kernels", fused_launch(g));
    g_launches = st == SGMV_OK ? launches + (S > 0 ? 2 : 1) : launches;
    return st;
}

int sgmv_debug_inject_wait_timeout(int enable) {
    g_inject_timeout = enable ? 1 : 0;
    return SGMV_OK;
}

int sgmv_read_floor(const void *src, size_t bytes, int32_t T, int32_t L, int32_t H1, int32_t H2,
                    int32_t r, int in_dtype, int y_dtype, int32_t *ctas, int32_t *cluster,
                    void *stream) {
    g_launches = 0;
    int st = check_common(T, L, r, 0, nullptr, nullptr, nullptr, in_dtype);
    if (st != SGMV_OK) return st;
    if ((st = check_dim(H1)) != SGMV_OK) return st;
    if ((st = check_dim(H2)) != SGMV_OK) return st;
    if (y_dtype != SGMV_F16 && y_dtype != SGMV_BF16 && y_dtype != SGMV_F32)
        return SGMV_ERR_INVALID_ARG;
    if (!src || bytes == 0 || T == 0) return SGMV_ERR_INVALID_ARG;
    if (!aligned16(src) || bytes % 16 != 0) return SGMV_ERR_ALIGNMENT;
    // the shape sgmv_apply_rows gives the streaming kernel for this batch:
    // the one-launch grouped form up to kGroupMaxT rows, else sgmv_apply on
    // the device grouping (sgmv_max_segments(T, L) segments, no host copy)
    const int32_t smax = sgmv_max_segments(T, L);
    StreamLaunch sl = {};
    if (!stream_shape(T, smax, nullptr, INT_MAX, H1, H2, r, in_dtype, y_dtype, sl,
                      T <= kGroupMaxT))
        return SGMV_ERR_UNSUPPORTED;
    int *err = error_word();
    if (!err) return SGMV_ERR_CUDA;
    const uint32_t chunk = sl.p.stage_bytes / 16u * 16u;
    st = cuda_status("read floor kernel",
                     read_floor_launch(src, (uint64_t)bytes, sl.p.cl, sl.p.G, sl.p.nst, chunk, err,
                                       static_cast<cudaStream_t>(stream)));
    if (st != SGMV_OK) return st;
    g_launches = 1;
    if (ctas) *ctas = sl.p.cl * sl.p.G;
    if (cluster) *cluster = sl.p.cl;
    return SGMV_OK;
}

int sgmv_get_device_error(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        note("cudaStreamSynchronize", e);
        return SGMV_ERR_CUDA;
    }
    int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_sgmv_error, sizeof(int))) != cudaSuccess) {
        note("read error word", e);
        return SGMV_ERR_CUDA;
    }
    if (v != 0) {
        const int zero = 0;
        if ((e = cudaMemcpyToSymbol(g_sgmv_error, &zero, sizeof(int))) != cudaSuccess) {
            note("clear error word", e);
            return SGMV_ERR_CUDA;
        }
    }
    return v;
}

}  // extern "C"
