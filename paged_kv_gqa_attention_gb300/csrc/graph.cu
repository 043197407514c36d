// Captured attention steps: a whole decode step (one qa_decode_attn per layer)
// or a whole prefill step of a packed bucket (one qa_prefill_attn per layer)
// captured once into a CUDA graph and replayed with a single launch.
//
// M* "Speech recognition: Whisper and Qwen3-ASR", "Serving notes": decode and
// prefill are captured per batch size / per packed bucket and replayed, so a
// step costs one launch instead of one per layer.  Every pointer, size and
// the workspace are fixed at capture; a replay reads whatever the buffers
// hold at that time, so the caller refills q, the page table, the lengths
// (and for prefill q/k/v and cu_seqlens) in place between replays.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <new>

#include "qa.h"
#include "qa_internal.h"

#define QA_API extern "C" __attribute__((visibility("default")))

struct qa_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int device = -1;
    int n_calls = 0;
};

namespace {

qa_status reject(qa_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
qa_status reject(qa_status st, const char *fmt, ...) {
    char msg[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(msg, sizeof msg, fmt, ap);
    va_end(ap);
    qa::set_last_error(msg);
    return st;
}

// Captures `n` calls of `call(i, stream)` on a private stream into a graph.
template <typename Call>
qa_status capture(const char *fn, int n, Call call, qa_graph **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: no CUDA device", fn);
    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: %s", fn, cudaGetErrorString(e));
    e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(s);
        return reject(QA_STATUS_LAUNCH_FAILED, "%s: %s", fn, cudaGetErrorString(e));
    }
    qa_status st = QA_STATUS_OK;
    char first_error[512] = "";
    for (int i = 0; i < n && st == QA_STATUS_OK; ++i) {
        st = call(i, s);
        if (st != QA_STATUS_OK) snprintf(first_error, sizeof first_error, "%s: call %d: %s", fn, i, qa_last_error());
    }
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(s, &g);
    cudaStreamDestroy(s);
    if (st != QA_STATUS_OK) {
        if (g) cudaGraphDestroy(g);
        qa::set_last_error(first_error);
        return st;
    }
    if (e != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: capture failed: %s", fn, cudaGetErrorString(e));
    cudaGraphExec_t x = nullptr;
    e = cudaGraphInstantiate(&x, g, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(g);
        return reject(QA_STATUS_LAUNCH_FAILED, "%s: instantiate failed: %s", fn, cudaGetErrorString(e));
    }
    qa_graph *h = new (std::nothrow) qa_graph;
    if (!h) {
        cudaGraphExecDestroy(x);
        cudaGraphDestroy(g);
        return reject(QA_STATUS_OOM, "%s: out of host memory", fn);
    }
    h->graph = g;
    h->exec = x;
    h->device = dev;
    h->n_calls = n;
    *out = h;
    return QA_STATUS_OK;
}

qa_status check_params(const char *fn, int n_layers, const qa_attn_params *p, qa_graph **out) {
    if (!out) return reject(QA_STATUS_INVALID_PARAMS, "%s: graph output pointer is NULL", fn);
    *out = nullptr;
    if (n_layers < 1) return reject(QA_STATUS_INVALID_PARAMS, "%s: n_layers %d < 1", fn, n_layers);
    if (!p) return reject(QA_STATUS_INVALID_PARAMS, "%s: params is NULL", fn);
    if (p->debug_checks)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: debug_checks synchronises and cannot be captured", fn);
    return QA_STATUS_OK;
}

}  // namespace

QA_API qa_status qa_decode_graph_create(int n_layers, const void *const *q, const void *const *k_pages,
                                        const void *const *v_pages, const int32_t *page_table,
                                        const int32_t *seq_lens, int batch, void *const *out,
                                        const qa_attn_params *params, qa_graph **graph) {
    const char *fn = "qa_decode_graph_create";
    qa::set_last_error("");
    qa_status st = check_params(fn, n_layers, params, graph);
    if (st != QA_STATUS_OK) return st;
    if (!q || !k_pages || !v_pages || !out) return reject(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer array", fn);
    return capture(
        fn, n_layers,
        [&](int i, cudaStream_t s) {
            qa_attn_params p = *params;
            p.stream = s;
            return qa_decode_attn(q[i], k_pages[i], v_pages[i], page_table, seq_lens, batch, out[i], &p);
        },
        graph);
}

QA_API qa_status qa_prefill_graph_create(int n_layers, const void *const *q, const void *const *k,
                                         const void *const *v, const int32_t *cu_seqlens, int batch,
                                         int total_tokens, const int32_t *page_table, void *const *k_pages,
                                         void *const *v_pages, void *const *out, const qa_attn_params *params,
                                         qa_graph **graph) {
    const char *fn = "qa_prefill_graph_create";
    qa::set_last_error("");
    qa_status st = check_params(fn, n_layers, params, graph);
    if (st != QA_STATUS_OK) return st;
    if (!q || !k || !v || !k_pages || !v_pages || !out)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: NULL pointer array", fn);
    return capture(
        fn, n_layers,
        [&](int i, cudaStream_t s) {
            qa_attn_params p = *params;
            p.stream = s;
            return qa_prefill_attn(q[i], k[i], v[i], cu_seqlens, batch, total_tokens, page_table, k_pages[i],
                                   v_pages[i], out[i], &p);
        },
        graph);
}

QA_API qa_status qa_graph_launch(qa_graph *graph, void *stream) {
    const char *fn = "qa_graph_launch";
    qa::set_last_error("");
    if (!graph || !graph->exec) return reject(QA_STATUS_INVALID_PARAMS, "%s: graph is NULL", fn);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != graph->device)
        return reject(QA_STATUS_INVALID_PARAMS, "%s: the graph was captured on device %d, current device is %d", fn,
                      graph->device, dev);
    const cudaError_t e = cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return reject(QA_STATUS_LAUNCH_FAILED, "%s: %s", fn, cudaGetErrorString(e));
    return QA_STATUS_OK;
}

QA_API void qa_graph_destroy(qa_graph *graph) {
    if (!graph) return;
    if (graph->exec) cudaGraphExecDestroy(graph->exec);
    if (graph->graph) cudaGraphDestroy(graph->graph);
    delete graph;
}
