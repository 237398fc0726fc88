/* A minimal NVTX tool for the tests: loaded by NVTX through the
 * NVTX_INJECTION64_PATH environment variable, it writes one line per
 * domain creation, range push and range pop to the file named by
 * FP8Q_NVTX_LOG.  Test code only. */
#include <stdio.h>
#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

static FILE* g_log;

static nvtxDomainHandle_t rec_domain_create(const char* name) {
  fprintf(g_log, "domain %s\n", name);
  fflush(g_log);
  return (nvtxDomainHandle_t)(void*)g_log;   /* any non-null handle */
}

static int rec_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t* a) {
  (void)d;
  fprintf(g_log, "push %s\n", a->messageType == NVTX_MESSAGE_TYPE_ASCII ? a->message.ascii : "?");
  fflush(g_log);
  return 0;
}

static int rec_pop(nvtxDomainHandle_t d) {
  (void)d;
  fprintf(g_log, "pop\n");
  fflush(g_log);
  return 0;
}

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
  const char* path = getenv("FP8Q_NVTX_LOG");
  if (!path || !(g_log = fopen(path, "w"))) return 0;
  const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
  if (!cb) return 0;
  NvtxFunctionTable table = 0;
  unsigned int size = 0;
  if (!cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &table, &size) || size < NVTX_CBID_CORE2_DomainCreateA)
    return 0;
  *table[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)rec_domain_create;
  *table[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)rec_push;
  *table[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)rec_pop;
  return 1;
}
