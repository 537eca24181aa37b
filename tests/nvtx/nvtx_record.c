/* Test aid: an NVTX injection library (loaded by NVTX through the
 * NVTX_INJECTION64_PATH environment variable) that appends every domain
 * creation, string registration, range push and range pop of the process to
 * the file named by NVTX_RECORD_PATH, one line each:
 *   domain <name> | push <domain> <name> <payload> | pop <domain>
 * Built from this source by the tracing test. */
#include <nvtx3/nvToolsExt.h>

#include <pthread.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static FILE* g_out;
static pthread_mutex_t g_mu = PTHREAD_MUTEX_INITIALIZER;

/* handles are heap copies of the names */
static nvtxDomainHandle_t NVTX_API rec_domain_create(const char* name) {
    pthread_mutex_lock(&g_mu);
    fprintf(g_out, "domain %s\n", name);
    fflush(g_out);
    pthread_mutex_unlock(&g_mu);
    return (nvtxDomainHandle_t)strdup(name);
}
static nvtxStringHandle_t NVTX_API rec_register_string(nvtxDomainHandle_t d, const char* s) {
    (void)d;
    return (nvtxStringHandle_t)strdup(s);
}
static int NVTX_API rec_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t* a) {
    const char* name = "?";
    if (a->messageType == NVTX_MESSAGE_TYPE_REGISTERED) name = (const char*)a->message.registered;
    else if (a->messageType == NVTX_MESSAGE_TYPE_ASCII) name = a->message.ascii;
    long long payload = a->payloadType == NVTX_PAYLOAD_TYPE_INT64 ? a->payload.llValue : 0;
    pthread_mutex_lock(&g_mu);
    fprintf(g_out, "push %s %s %lld\n", d ? (const char*)d : "-", name, payload);
    fflush(g_out);
    pthread_mutex_unlock(&g_mu);
    return 0;
}
static int NVTX_API rec_pop(nvtxDomainHandle_t d) {
    pthread_mutex_lock(&g_mu);
    fprintf(g_out, "pop %s\n", d ? (const char*)d : "-");
    fflush(g_out);
    pthread_mutex_unlock(&g_mu);
    return 0;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
    const char* path = getenv("NVTX_RECORD_PATH");
    if (!path || !(g_out = fopen(path, "a"))) return 0;
    const NvtxExportTableCallbacks* cb =
        (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &table, &size) || !table ||
        size <= NVTX_CBID_CORE2_DomainCreateA)
        return 0;
    *table[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)rec_domain_create;
    *table[NVTX_CBID_CORE2_DomainRegisterStringA] = (NvtxFunctionPointer)rec_register_string;
    *table[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)rec_push;
    *table[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)rec_pop;
    return 1;
}
