// sgmv_builder.cu -- device kernel that groups a batch's rows by adapter id.
//
// The batch builder groups requests by LoRA id ("Punica: when LoRA
// fine-tuned models need multi-tenant serving", omica.com.cn article, §5.1)
// and SGMV runs over the resulting contiguous segments ("Punica: Multi-Tenant
// LoRA Serving", nubint.ai review, "Proposed method").  Here the grouping is
// a stable counting sort on the GPU: ascending id with -1 (no adapter) first,
// original row order inside an id.
//
// One CTA of 1024 threads:
//   1. histogram of ids in shared memory (bin b holds id b-1);
//   2. block scan of the bins: start position of each id and segment number
//      of each id that occurs;
//   3. griddepcontrol.wait -- the outputs may still be read by the SGMV kernel
//      launched before on the stream -- then write seg_ptr / idx and pad them
//      with empty segments up to S_max;
//   4. stable scatter of row numbers into perm, 32 rows per step per warp,
//      ranking equal ids inside a step with __match_any_sync: for large
//      batches every warp takes a contiguous chunk of rows, placed from
//      per-(warp, id) start positions; otherwise one warp walks all rows.
// The kernel never triggers its dependents early, so the next kernel on the
// stream starts only after the metadata is complete.
#include "sgmv_device.cuh"
#include "sgmv_internal.h"

namespace sgmv {

constexpr int kBuilderThreads = 1024;

__global__ void __launch_bounds__(kBuilderThreads)
    build_segments_kernel(const int32_t *__restrict__ ra, int32_t T, int32_t L,
                          int32_t *__restrict__ perm, int32_t *__restrict__ seg_ptr,
                          int32_t *__restrict__ idx, int32_t *__restrict__ S_out, int32_t S_max,
                          int *err, bool multi_warp) {
    extern __shared__ int cnt[];  // L + 1 bins (then the per-warp table when multi_warp)
    __shared__ int w_c[32], w_n[32];
    __shared__ int s_total;
    const int nb = L + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;

    for (int b = tid; b < nb; b += blockDim.x) cnt[b] = 0;
    __syncthreads();
    for (int t = tid; t < T; t += blockDim.x) {
        int key = ra[t] + 1;
        if (key < 0 || key > L) {
            set_error(err, kErrBadIndex);
            key = 0;
        }
        atomicAdd(&cnt[key], 1);
    }
    __syncthreads();

    // Each thread owns a contiguous run of bins.
    const int per = (nb + blockDim.x - 1) / blockDim.x;
    const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
    int c_own = 0, n_own = 0;
    for (int b = b0; b < b1; ++b) {
        c_own += cnt[b];
        n_own += cnt[b] > 0;
    }
    int c_in = c_own, n_in = n_own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int c = __shfl_up_sync(0xffffffffu, c_in, off);
        const int n = __shfl_up_sync(0xffffffffu, n_in, off);
        if (lane >= off) {
            c_in += c;
            n_in += n;
        }
    }
    if (lane == 31) {
        w_c[warp] = c_in;
        w_n[warp] = n_in;
    }
    __syncthreads();
    if (warp == 0) {
        const int c = lane < nwarps ? w_c[lane] : 0;
        const int n = lane < nwarps ? w_n[lane] : 0;
        int ci = c, ni = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int cc = __shfl_up_sync(0xffffffffu, ci, off);
            const int nn = __shfl_up_sync(0xffffffffu, ni, off);
            if (lane >= off) {
                ci += cc;
                ni += nn;
            }
        }
        w_c[lane] = ci - c;
        w_n[lane] = ni - n;
        if (lane == 31) s_total = ni;
    }
    __syncthreads();
    int pos = w_c[warp] + c_in - c_own;  // first sorted position of this thread's bins
    int sid = w_n[warp] + n_in - n_own;  // segment number of its first non-empty bin
    const int S = s_total;

    pdl_wait();

    for (int b = b0; b < b1; ++b) {
        const int c = cnt[b];
        if (c > 0) {
            seg_ptr[sid] = pos;
            idx[sid] = b - 1;
            ++sid;
        }
        cnt[b] = pos;  // from here on: next free position of the bin
        pos += c;
    }
    if (tid == 0) {
        seg_ptr[S] = T;
        *S_out = S;
    }
    for (int s = S + tid; s < S_max; s += blockDim.x) {
        idx[s] = -1;
        seg_ptr[s + 1] = T;
    }
    __syncthreads();

    // Stable scatter.  With a per-warp table (multi_warp), the rows are cut
    // into one contiguous chunk per warp: each warp counts its chunk's ids,
    // the counts are turned into per-(warp, id) start positions, and every
    // warp places its chunk in order.  Otherwise one warp walks all rows.
    const int nw = multi_warp ? nwarps : 1;
    const int chunk = (T + nw - 1) / nw;
    int *wpos = cnt + nb;  // [nwarps][nb], multi_warp only
    if (multi_warp) {
        for (int e = tid; e < nwarps * nb; e += blockDim.x) wpos[e] = 0;
        __syncthreads();
        for (int t = warp * chunk + lane; t < min(T, (warp + 1) * chunk); t += 32) {
            int key = ra[t] + 1;
            if (key < 0 || key > L) key = 0;
            atomicAdd(&wpos[warp * nb + key], 1);
        }
        __syncthreads();
        for (int b = tid; b < nb; b += blockDim.x) {
            int off = cnt[b];
            for (int w = 0; w < nwarps; ++w) {
                const int c = wpos[w * nb + b];
                wpos[w * nb + b] = off;
                off += c;
            }
        }
        __syncthreads();
    }
    if (warp < nw) {
        int *run = multi_warp ? wpos + warp * nb : cnt;
        const int t_end = min(T, (warp + 1) * chunk);
        for (int base = warp * chunk; base < t_end; base += 32) {
            const int t = base + lane;
            int key = -1;  // lanes past the chunk get a key no real row has
            if (t < t_end) {
                key = ra[t] + 1;
                if (key < 0 || key > L) key = 0;
            }
            const unsigned grp = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(grp & ((1u << lane) - 1u));
            if (t < t_end) perm[run[key] + rank] = t;
            __syncwarp();
            if (t < t_end && rank == 0) run[key] += __popc(grp);
            __syncwarp();
        }
    }
}

int build_segments_launch(const int32_t *row_adapter, int32_t T, int32_t L, int32_t *perm,
                          int32_t *seg_ptr, int32_t *idx, int32_t *S, int32_t S_max, int *err,
                          cudaStream_t stream) {
    // per-warp table when it fits in 96 KB next to the bins and there are
    // enough rows to share out
    const bool multi_warp = T > 256 && (size_t)(L + 1) * (kBuilderThreads / 32 + 1) * 4 <= 98304;
    const size_t smem = (size_t)(L + 1) * sizeof(int) * (multi_warp ? kBuilderThreads / 32 + 1 : 1);
    cudaError_t e = cudaFuncSetAttribute(build_segments_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kBuilderThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, build_segments_kernel, row_adapter, T, L, perm, seg_ptr,
                                   idx, S, S_max, err, multi_warp);
}

}  // namespace sgmv
