// kda_prefill_tc_precise.cu -- the tensor-core prefill compiled in its precise mode, for
// kda_prefill_precise: the output product's A operand Aqk carried as fp16(Aqk) plus its low part,
// so that P = Aqk Bt is not limited by one fp16 rounding of Aqk.  Everything else is the default
// kernel ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA", second
// paragraph: chunked prefill with tile products on the tensor cores).
#define KDA_PRECISE 1
#include "kda_prefill_tc.cu"
