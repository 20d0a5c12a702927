#define PA_D 64
#include "pa_decode_inst.inc"
