/* A minimal NVTX tool for the tests. The NVTX runtime of a library loads it from
 * NVTX_INJECTION64_PATH and calls InitializeInjectionNvtx2, which installs three
 * callbacks: domain creation, and push and pop of a domain range. It records
 * "domain/name" for every range pushed and counts the pops, so a test can check which
 * calls a library traces and that every range it opens is closed. No GPU is involved. */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#define MAX_DOMAINS 64

static char g_ranges[1 << 16];
static size_t g_ranges_len;
static const char *g_domain_names[MAX_DOMAINS];
static char g_domain_store[MAX_DOMAINS][64];
static int g_n_domains;
static int g_pushes, g_pops, g_depth, g_min_depth;

static void append(const char *a, const char *b)
{
    const size_t na = strlen(a), nb = strlen(b);
    if (g_ranges_len + na + nb + 3 > sizeof g_ranges) return;
    memcpy(g_ranges + g_ranges_len, a, na);
    g_ranges_len += na;
    g_ranges[g_ranges_len++] = '/';
    memcpy(g_ranges + g_ranges_len, b, nb);
    g_ranges_len += nb;
    g_ranges[g_ranges_len++] = '\n';
    g_ranges[g_ranges_len] = 0;
}

/* handles are 1-based indices into the domain table */
static nvtxDomainHandle_t NVTX_API rec_domain_create(const char *name)
{
    if (g_n_domains >= MAX_DOMAINS) return (nvtxDomainHandle_t)0;
    strncpy(g_domain_store[g_n_domains], name ? name : "?", sizeof g_domain_store[0] - 1);
    g_domain_names[g_n_domains] = g_domain_store[g_n_domains];
    ++g_n_domains;
    return (nvtxDomainHandle_t)(uintptr_t)g_n_domains;
}

static const char *domain_name(nvtxDomainHandle_t d)
{
    const uintptr_t i = (uintptr_t)d;
    return (i >= 1 && i <= (uintptr_t)g_n_domains) ? g_domain_names[i - 1] : "?";
}

static int NVTX_API rec_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t *a)
{
    const char *msg = (a && a->messageType == NVTX_MESSAGE_TYPE_ASCII && a->message.ascii) ? a->message.ascii : "?";
    append(domain_name(d), msg);
    ++g_pushes;
    return g_depth++;
}

static int NVTX_API rec_pop(nvtxDomainHandle_t d)
{
    (void)d;
    ++g_pops;
    --g_depth;
    if (g_depth < g_min_depth) g_min_depth = g_depth;
    return g_depth;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table)
{
    const NvtxExportTableCallbacks *cb = (const NvtxExportTableCallbacks *)get_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = NULL;
    unsigned int last = 0;        /* highest valid callback index of the module */
    if (!cb || !cb->GetModuleFunctionTable || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE2, &table, &last))
        return 0;
    if (!table || last < NVTX_CBID_CORE2_DomainCreateA) return 0;
    *table[NVTX_CBID_CORE2_DomainRangePushEx] = (NvtxFunctionPointer)rec_push;
    *table[NVTX_CBID_CORE2_DomainRangePop] = (NvtxFunctionPointer)rec_pop;
    *table[NVTX_CBID_CORE2_DomainCreateA] = (NvtxFunctionPointer)rec_domain_create;
    return 1;
}

const char *nvtx_recorder_ranges(void) { return g_ranges; }
int nvtx_recorder_pushes(void) { return g_pushes; }
int nvtx_recorder_pops(void) { return g_pops; }
int nvtx_recorder_min_depth(void) { return g_min_depth; }
