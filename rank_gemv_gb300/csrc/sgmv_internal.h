// sgmv_internal.h -- parameters shared by the C-ABI host code and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (no libcuda link)
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgmv {

// Which part of SGMV a CUDA-core launch runs.
enum Mode : int {
    kFused = 0,   // shrink + expand, v kept in shared memory of a cluster
    kShrink = 1,  // shrink only, v written to device memory
    kExpand = 2,  // expand only, v read from device memory
    kGrouped = 3, // kFused, each CTA grouping the rows itself from row_adapter
};

// Largest batch kGrouped handles.  Each CTA spends O(T) shared-memory steps
// per row on the grouping, which stops paying off against reading
// precomputed metadata beyond a few dozen rows.
constexpr int kGroupMaxT = 64;

constexpr int kThreads = 256;   // threads per CTA of the CUDA-core kernels
constexpr int kRowsMax = 8;     // rows of one segment handled by one tile
constexpr int kStageBytes = 32768;  // bytes of one staged chunk (A+X or B)

// One CUDA-core launch.  Grid: x = slice of H1 (and H2) owned by one CTA, or
// of H2 alone in kExpand; y = tile slot.  A tile is up to `rows` consecutive
// sorted positions of one segment.  In kFused / kShrink the CTAs along x form
// one thread-block cluster and reduce their partial v through distributed
// shared memory.
struct CCParams {
    void *y;
    const void *x;
    const void *A;
    const void *B;
    const float *v_in;   // kExpand: v [T][r]
    float *v_out;        // kShrink: v [T][r]
    const int32_t *perm;
    const int32_t *seg_ptr;
    const int32_t *idx;
    int *err;            // sticky device error word
    const int32_t *row_adapter;  // kGrouped: adapter id of every row
    int32_t *perm_out;           // kGrouped, optional: grouping written out
    int32_t *seg_out;
    int32_t *idx_out;
    int32_t *S_out;
    int32_t S_max;
    int32_t S, T, L, H1, H2, r;
    int32_t rows;        // rows per tile, 1..kRowsMax
    int32_t hc, jc;      // columns of H1 / H2 owned by one CTA (multiples of 8)
    int32_t hs, js;      // columns staged in shared memory at once (multiples of 8)
    int32_t ax_stages;   // 1 or 2 buffers for (A, X) chunks
    int32_t b_stages;    // 1 or 2 buffers for B chunks
    int32_t cl;          // CTAs per cluster along x (1 = no cluster)
    int32_t rmax;        // compile-time bound on r of the launched kernel
    int32_t ysize;       // bytes per element of y
    int32_t y_pref;      // 1: the CTA's y rows are prefetched into shared memory
    int32_t min_len;     // only segments with min_len <= length <= max_len
    int32_t max_len;
    float scale;
};

struct CCSmem {
    uint32_t ax_stage_bytes, b_stage_bytes, ax_off, b_off, y_off, recv_off, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Dynamic shared memory of a CUDA-core launch; identical on host and device.
__host__ __device__ inline CCSmem cc_smem_layout(const CCParams &p, int elem, int mode) {
    CCSmem s;
    const bool ax = mode != kExpand, b = mode != kShrink;
    s.ax_stage_bytes = ax ? align_up((uint32_t)(p.hs * p.r + p.rows * p.hs) * elem, 128) : 0;
    s.b_stage_bytes = b ? align_up((uint32_t)(p.r * p.js) * elem, 128) : 0;
    s.ax_off = 0;
    s.b_off = ax ? s.ax_stage_bytes * p.ax_stages : 0;
    // y rows of the tile: [rows][jc] when the CTA's whole H2 slice is one chunk
    s.y_off = s.b_off + (b ? s.b_stage_bytes * p.b_stages : 0);
    const uint32_t y_bytes = (b && p.y_pref) ? align_up((uint32_t)(p.rows * p.jc * p.ysize), 128) : 0;
    // partial v of every CTA of the cluster: [cl][kRowsMax][rmax] fp32
    s.recv_off = s.y_off + y_bytes;
    const uint32_t recv_bytes = (ax && p.cl > 1) ? (uint32_t)(p.cl * kRowsMax * p.rmax) * 4u : 0;
    s.total = s.recv_off + recv_bytes;
    return s;
}

struct CCLaunch {
    CCParams p;
    int mode;
    int y_dtype;   // SGMV_F16 / SGMV_BF16 / SGMV_F32
    int rmax;      // 16, 32, 64 or 128: compile-time bound on r
    dim3 grid;
    int cluster;   // CTAs per cluster along x (1 = plain launch)
    cudaStream_t stream;
    bool pdl;
};

// Tensor-core launch pair (shrink then expand) for segments of at least
// min_len rows.  v is kept in the workspace as two 16-bit halves, vhi and vlo.
struct TCArgs {
    void *y;
    const void *x;
    const void *A;
    const void *B;
    const int32_t *perm;
    const int32_t *seg_ptr;
    const int32_t *idx;
    int *err;
    void *vhi;
    void *vlo;
    int32_t S, T, L, H1, H2, r;
    int32_t min_len, max_len;
    float scale;
    int in_dtype, y_dtype;
    int64_t slots;   // 128-row tile slots
    int32_t nsm;     // streaming multiprocessors of the device
    cudaStream_t stream;
};

// Segments at least this long go to the tensor cores (when a workspace is
// given and r is 64 or 128).
constexpr int kTcMinLen = 64;

int tc_launch(const TCArgs &g);

// Encode a tiled tensor map (f16 / bf16 elements, 128-byte swizzle or none).
bool tmap_encode(CUtensorMap *m, bool bf16, int rank, const void *ptr, const cuuint64_t *dims,
                 const cuuint64_t *strides, const cuuint32_t *box, bool swizzle128);

// Launch one CUDA-core kernel; returns a cudaError_t value.
int cc_launch_f16(const CCLaunch &l);
int cc_launch_bf16(const CCLaunch &l);

// Launch the device grouping kernel; returns a cudaError_t value.
int build_segments_launch(const int32_t *row_adapter, int32_t T, int32_t L, int32_t *perm,
                          int32_t *seg_ptr, int32_t *idx, int32_t *S, int32_t S_max, int *err,
                          cudaStream_t stream);


// ---- persistent streaming CUDA-core kernel (short segments, r <= 64) -------
// Compute warps per CTA: 8 (two CTAs fit on an SM), or 16 when one CTA owns
// whole tiles and a whole SM; plus one copy-issuing warp.
constexpr int kStreamMaxStages = 8;
constexpr int kStreamMaxTiles = 64;   // tiles one cluster walks in one launch
// Columns of one A chunk and of one B chunk at rank bound RK (32 KB of
// weights per chunk at r = RK): 1024 for RK = 16, 512 for RK = 32.
constexpr int kStreamChunkElems = 16384;

// One launch of the streaming kernel.  Grid: x = CTA rank in the cluster
// (slices [rank*hc, ...) of H1 and [rank*jc, ...) of H2), y = cluster; cluster
// c walks the tiles c, c + G, c + 2G, ... of the batch.  Every CTA streams its
// slices of the tiles' A and B through a ring of `nst` shared-memory stages.
// Most problems (same rows and segments, own x, A, B and y) in one launch of
// the streaming kernel.
constexpr int kStreamMaxProblems = 4;

// Everything of a launch but the problems' operands.
struct StreamCommon {
    int32_t b4d;                 // B read as whole chunks through a 4-D view (below)
    int32_t np;                  // problems: 1 .. kStreamMaxProblems (1 in the grouped form)
    const int32_t *perm;
    const int32_t *seg_ptr;
    const int32_t *idx;
    int *err;
    const int32_t *row_adapter;  // grouped form: adapter id of every row
    int32_t *perm_out;           // grouped form, optional: grouping written out
    int32_t *seg_out;
    int32_t *idx_out;
    int32_t *S_out;
    int32_t S_max;
    int32_t S, T, L, H1, H2, r;
    int32_t cl, G;               // CTAs per cluster, clusters
    int32_t hc, jc;              // columns of H1 / H2 per CTA (multiples of 8)
    int32_t hn;                  // columns of one A or B chunk (kStreamChunkElems / rank bound)
    int32_t nst;                 // ring stages
    int32_t trows;               // rows per tile, 1..8 (the x / y part of a stage holds trows rows)
    uint32_t stage_bytes, act_off;  // bytes per stage; offset of the x / y rows in it
    uint32_t red_off, recv_off, v_off, tab_off, smem_bytes;
    int32_t min_len, max_len;
    float scale;
    int32_t inject;              // 1: diagnostic launch with an injected wait timeout
};

// The operands of NP problems.
template <int NP> struct StreamOperands {
    // B of each problem, no swizzle: as [L][H2/256][r][256] with box
    // {256, r, chunk/256, 1} (b4d, whole chunk in one copy), else as
    // [L][r][H2] with box {256, r, 1}
    CUtensorMap tmap_b[NP];
    void *y[NP];
    const void *x[NP];
    const void *A[NP];
    const void *B[NP];
};

// The parameters with the operands of NP problems (first, so that the tensor
// maps open the parameter block).  The kernel for one problem takes NP = 1:
// its parameter block is 400 bytes smaller, which measured 1-2 % faster per
// call on decode batches.
template <int NP> struct StreamParamsT : StreamOperands<NP>, StreamCommon {};
using StreamParams = StreamParamsT<kStreamMaxProblems>;  // what the host fills
using StreamParams1 = StreamParamsT<1>;

struct StreamLaunch {
    StreamParams p;
    int in_dtype, y_dtype;
    int rk;          // 16, 32 or 64: compile-time bound on r
    int cw;          // compute warps: 8 or 16
    bool grouped;
    bool multi;      // the instantiation for several problems (one-CTA clusters, cw 16)
    cudaStream_t stream;
};

// Launch the streaming kernel; returns a cudaError_t value.
int stream_launch_f16(const StreamLaunch &l);
int stream_launch_bf16(const StreamLaunch &l);

// Launch shape of the streaming kernel for np problems of these shapes (see
// sgmv_api.cu); false when the kernel does not apply.
bool stream_shape(int32_t T, int32_t S, const int32_t *seg_ptr_host, int32_t max_len, int32_t H1,
                  int32_t H2, int32_t r, int in_dtype, int y_dtype, StreamLaunch &l,
                  bool grouped, int np = 1);

// Read-only kernel with a given grid, cluster size and ring (sgmv_floor.cu);
// returns a cudaError_t value.
int read_floor_launch(const void *src, uint64_t bytes, int cl, int G, int nst, uint32_t chunk,
                      int *err, cudaStream_t stream);


// Records a failed CUDA call for sgmv_last_error_string (calling thread).
void note_cuda_error(const char *what, cudaError_t e);

// Sticky device error word of the current device, or nullptr (error noted).
int *device_error_word();

}  // namespace sgmv
