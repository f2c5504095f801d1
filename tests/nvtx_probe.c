/* nvtx_probe.c -- a minimal NVTX injection library for the tests: it takes over the core
 * nvtxRangePushA / nvtxRangePop callbacks and records each as one line ("+name" or "-") in a
 * buffer that the test reads back with nvtx_probe_log().  Loaded by the NVTX headers inside
 * libmamba_state.so when NVTX_INJECTION64_PATH names this library. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

typedef void (*fnptr_t)(void);
typedef int (*get_module_table_t)(int module, fnptr_t ***table, unsigned int *size);
typedef struct {
    size_t struct_size;
    get_module_table_t get_module_function_table;
} callbacks_table_t;
typedef const void *(*get_export_table_t)(uint32_t id);

enum { ETID_CALLBACKS = 1, MODULE_CORE = 1, CBID_RANGE_PUSH_A = 9, CBID_RANGE_POP = 11 };

static char g_log[1 << 16];
static size_t g_len;

static void append(const char *s) {
    size_t n = strlen(s);
    if (g_len + n + 1 < sizeof(g_log)) {
        memcpy(g_log + g_len, s, n);
        g_len += n;
        g_log[g_len++] = '\n';
        g_log[g_len] = 0;
    }
}

static int on_push(const char *name) {
    char line[256];
    snprintf(line, sizeof line, "+%s", name ? name : "");
    append(line);
    return 0;
}

static int on_pop(void) {
    append("-");
    return 0;
}

int InitializeInjectionNvtx2(get_export_table_t get_export_table) {
    const callbacks_table_t *cb = (const callbacks_table_t *)get_export_table(ETID_CALLBACKS);
    fnptr_t **table = 0;
    unsigned int size = 0;
    if (!cb || !cb->get_module_function_table(MODULE_CORE, &table, &size) || size <= CBID_RANGE_POP) return 0;
    *table[CBID_RANGE_PUSH_A] = (fnptr_t)on_push;
    *table[CBID_RANGE_POP] = (fnptr_t)on_pop;
    return 1;
}

const char *nvtx_probe_log(void) { return g_log; }
void nvtx_probe_clear(void) { g_len = 0; g_log[0] = 0; }
