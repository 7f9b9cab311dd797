/* Output encodings of the synthetic generator's fills. */
#ifndef SYNTH_KINDS_H
#define SYNTH_KINDS_H
enum {
  SYNTH_OUT_F32 = 0,         /* fp32 value                                   */
  SYNTH_OUT_BF16 = 1,        /* bfloat16 bits, fp32 value truncated          */
  SYNTH_OUT_F16 = 2,         /* binary16 bits, fp32 value truncated          */
  SYNTH_OUT_F32_OF_BF16 = 3, /* fp32 holding exactly the truncated bfloat16  */
  SYNTH_OUT_F32_OF_F16 = 4   /* fp32 holding exactly the truncated binary16  */
};
#endif
