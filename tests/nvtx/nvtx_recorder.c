/* nvtx_recorder.c -- a minimal NVTX tool for the tests: loaded through NVTX_INJECTION64_PATH,
 * it appends the name of every range pushed with nvtxRangePushA (and a line per pop) to the
 * file named by FCM_NVTX_LOG.  Built by tests/test_nvtx.py with the host compiler. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE *g_log;

static int NVTX_API push_a(const char *name) {
    if (g_log) {
        fprintf(g_log, "push %s\n", name ? name : "");
        fflush(g_log);
    }
    return 0;
}

static int NVTX_API pop(void) {
    if (g_log) {
        fputs("pop\n", g_log);
        fflush(g_log);
    }
    return 0;
}

__attribute__((visibility("default"))) int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get) {
    const char *path = getenv("FCM_NVTX_LOG");
    if (!path || !get) return 0;
    g_log = fopen(path, "a");
    const NvtxExportTableCallbacks *cb = (const NvtxExportTableCallbacks *)get(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!g_log || !cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
    if (size <= NVTX_CBID_CORE_RangePop) return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)push_a;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)pop;
    return 1;
}
