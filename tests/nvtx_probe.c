/* nvtx_probe.c — a minimal NVTX tool for the tests: loaded through
 * NVTX_INJECTION64_PATH, it records every domain created and every range
 * pushed and popped (name, int64 payload, domain name, nesting depth, thread)
 * so that a test can read back, through ctypes, which ranges the library
 * emitted and in what order.
 *
 * NVTX's loadable-tool protocol: the NVTX headers compiled into a library
 * look up InitializeInjectionNvtx2 in the tool on their first call and hand
 * it a function that returns export tables; the callbacks table gives the
 * tool each module's table of function pointers, which the tool overwrites
 * with its own handlers.  Every library that carries its own copy of the
 * NVTX headers initialises separately, so the tool may be initialised more
 * than once; it patches every table it is given.  Only the domain calls are
 * recorded (the library's ranges are all in its own domain).
 */
#include <nvtx3/nvToolsExt.h>

#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PROBE_MAX 65536
#define PROBE_NAME 48
#define PROBE_DOMAINS 32

typedef struct {
  int32_t kind; /* 1 push, 2 pop */
  int32_t depth; /* nesting depth on its thread before the push / after the pop */
  int32_t domain; /* index into the domain names, -1 if unknown */
  int64_t payload;
  uint64_t thread;
  char name[PROBE_NAME];
} probe_event;

static pthread_mutex_t g_mu = PTHREAD_MUTEX_INITIALIZER;
static probe_event g_ev[PROBE_MAX];
static int64_t g_n, g_dropped;
static char g_domain[PROBE_DOMAINS][PROBE_NAME];
static int32_t g_n_domains;
static int32_t g_inits;
static __thread int32_t t_depth;

static int32_t domain_index(nvtxDomainHandle_t d) {
  const intptr_t i = (intptr_t)d - 1;
  return (d && i >= 0 && i < g_n_domains) ? (int32_t)i : -1;
}

static void record(int32_t kind, int32_t depth, nvtxDomainHandle_t d,
                   const nvtxEventAttributes_t* a) {
  pthread_mutex_lock(&g_mu);
  if (g_n >= PROBE_MAX) {
    g_dropped++;
  } else {
    probe_event* e = &g_ev[g_n++];
    memset(e, 0, sizeof(*e));
    e->kind = kind;
    e->depth = depth;
    e->domain = domain_index(d);
    e->thread = (uint64_t)pthread_self();
    if (a && a->payloadType == NVTX_PAYLOAD_TYPE_INT64) e->payload = a->payload.llValue;
    if (a && a->messageType == NVTX_MESSAGE_TYPE_ASCII && a->message.ascii)
      strncpy(e->name, a->message.ascii, PROBE_NAME - 1);
  }
  pthread_mutex_unlock(&g_mu);
}

static nvtxDomainHandle_t NVTX_API probe_domain_create(const char* name) {
  pthread_mutex_lock(&g_mu);
  int32_t i;
  for (i = 0; i < g_n_domains; ++i)
    if (strncmp(g_domain[i], name, PROBE_NAME - 1) == 0) break;
  if (i == g_n_domains && g_n_domains < PROBE_DOMAINS) {
    strncpy(g_domain[i], name, PROBE_NAME - 1);
    g_n_domains++;
  }
  pthread_mutex_unlock(&g_mu);
  return i < PROBE_DOMAINS ? (nvtxDomainHandle_t)(intptr_t)(i + 1) : (nvtxDomainHandle_t)0;
}

static int NVTX_API probe_domain_push(nvtxDomainHandle_t d, const nvtxEventAttributes_t* a) {
  record(1, t_depth, d, a);
  return t_depth++;
}

static int NVTX_API probe_domain_pop(nvtxDomainHandle_t d) {
  --t_depth;
  record(2, t_depth, d, 0);
  return t_depth;
}

static int patch(const NvtxExportTableCallbacks* cb, NvtxCallbackModule m, unsigned id,
                 NvtxFunctionPointer f) {
  NvtxFunctionTable table = 0;
  unsigned size = 0;
  if (!cb->GetModuleFunctionTable(m, &table, &size) || !table || id >= size || !table[id])
    return 0;
  *table[id] = f;
  return 1;
}

int NVTX_API InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get) {
  const NvtxExportTableCallbacks* cb =
      (const NvtxExportTableCallbacks*)get(NVTX_ETID_CALLBACKS);
  if (!cb || cb->struct_size < sizeof(NvtxExportTableCallbacks)) return 0;
  int ok = 1;
  ok &= patch(cb, NVTX_CB_MODULE_CORE2, NVTX_CBID_CORE2_DomainCreateA,
              (NvtxFunctionPointer)probe_domain_create);
  ok &= patch(cb, NVTX_CB_MODULE_CORE2, NVTX_CBID_CORE2_DomainRangePushEx,
              (NvtxFunctionPointer)probe_domain_push);
  ok &= patch(cb, NVTX_CB_MODULE_CORE2, NVTX_CBID_CORE2_DomainRangePop,
              (NvtxFunctionPointer)probe_domain_pop);
  pthread_mutex_lock(&g_mu);
  g_inits++;
  pthread_mutex_unlock(&g_mu);
  return ok;
}

/* ---- read-back, through ctypes ---- */

int64_t probe_count(void) { return g_n; }
int64_t probe_dropped(void) { return g_dropped; }
int32_t probe_inits(void) { return g_inits; }

int32_t probe_event_at(int64_t i, int32_t* kind, int32_t* depth, int64_t* payload,
                       uint64_t* thread, char* name, char* domain) {
  pthread_mutex_lock(&g_mu);
  if (i < 0 || i >= g_n) {
    pthread_mutex_unlock(&g_mu);
    return 0;
  }
  const probe_event* e = &g_ev[i];
  *kind = e->kind;
  *depth = e->depth;
  *payload = e->payload;
  *thread = e->thread;
  memcpy(name, e->name, PROBE_NAME);
  memset(domain, 0, PROBE_NAME);
  if (e->domain >= 0) memcpy(domain, g_domain[e->domain], PROBE_NAME);
  pthread_mutex_unlock(&g_mu);
  return 1;
}

void probe_reset(void) {
  pthread_mutex_lock(&g_mu);
  g_n = 0;
  g_dropped = 0;
  pthread_mutex_unlock(&g_mu);
}
