// tmem_fold.cuh: acc[0..127] += sc * (128 consecutive fp32 TMEM columns of
// this thread's lane), as ONE inline-asm statement, in two forms.
//
// Four 32-column tcgen05.ld loads; each load after the first is issued before
// the previous chunk's FMAs, so the TMEM read latency overlaps arithmetic,
// and the temporaries live only inside the statement (the compiler cannot
// stretch their lifetimes across chunks).  `taddr` is the TMEM address of
// column 0 (lane field set by the caller), `sc` the per-row block-scale
// product.  The statements are spelled out in full: four loads into two banks
// of 32 registers (t0-31, t32-63), then the FMAs.
//
// tmem_fold128 keeps 128 fp32 accumulators and folds with fma.rn.f32.
// tmem_fold128x2 keeps them as 64 packed pairs (column 2i in the low half of
// acc[i], 2i+1 in the high half) and folds with the packed fma.rn.f32x2: two
// independent fp32 FMAs, each rounded like fma.rn.f32, so the sums are
// bit-for-bit the same with half the FMA instructions.  Which one is faster
// depends on the kernel around it (the standalone GEMM1: the packed form by
// 4%; the fused stage1 kernel: the scalar form by 3%, measured on one box).
// tmem_fold32x2 and tmem_fold32 (at the end) fold the transposed units of few
// rows, in the packed and the scalar form.
#pragma once

#include "common.cuh"

namespace moe {

MOE_DEV void tmem_fold128(uint32_t taddr, float sc, float (&acc)[128]) {
  asm volatile(
      "{\n\t.reg .b32 t<64>;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%128+0];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%128+32];\n\t"
      "fma.rn.f32 %0, t0, %129, %0; fma.rn.f32 %1, t1, %129, %1; fma.rn.f32 %2, t2, %129, %2; fma.rn.f32 %3, t3, %129, %3;\n\t"
      "fma.rn.f32 %4, t4, %129, %4; fma.rn.f32 %5, t5, %129, %5; fma.rn.f32 %6, t6, %129, %6; fma.rn.f32 %7, t7, %129, %7;\n\t"
      "fma.rn.f32 %8, t8, %129, %8; fma.rn.f32 %9, t9, %129, %9; fma.rn.f32 %10, t10, %129, %10; fma.rn.f32 %11, t11, %129, %11;\n\t"
      "fma.rn.f32 %12, t12, %129, %12; fma.rn.f32 %13, t13, %129, %13; fma.rn.f32 %14, t14, %129, %14; fma.rn.f32 %15, t15, %129, %15;\n\t"
      "fma.rn.f32 %16, t16, %129, %16; fma.rn.f32 %17, t17, %129, %17; fma.rn.f32 %18, t18, %129, %18; fma.rn.f32 %19, t19, %129, %19;\n\t"
      "fma.rn.f32 %20, t20, %129, %20; fma.rn.f32 %21, t21, %129, %21; fma.rn.f32 %22, t22, %129, %22; fma.rn.f32 %23, t23, %129, %23;\n\t"
      "fma.rn.f32 %24, t24, %129, %24; fma.rn.f32 %25, t25, %129, %25; fma.rn.f32 %26, t26, %129, %26; fma.rn.f32 %27, t27, %129, %27;\n\t"
      "fma.rn.f32 %28, t28, %129, %28; fma.rn.f32 %29, t29, %129, %29; fma.rn.f32 %30, t30, %129, %30; fma.rn.f32 %31, t31, %129, %31;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%128+64];\n\t"
      "fma.rn.f32 %32, t32, %129, %32; fma.rn.f32 %33, t33, %129, %33; fma.rn.f32 %34, t34, %129, %34; fma.rn.f32 %35, t35, %129, %35;\n\t"
      "fma.rn.f32 %36, t36, %129, %36; fma.rn.f32 %37, t37, %129, %37; fma.rn.f32 %38, t38, %129, %38; fma.rn.f32 %39, t39, %129, %39;\n\t"
      "fma.rn.f32 %40, t40, %129, %40; fma.rn.f32 %41, t41, %129, %41; fma.rn.f32 %42, t42, %129, %42; fma.rn.f32 %43, t43, %129, %43;\n\t"
      "fma.rn.f32 %44, t44, %129, %44; fma.rn.f32 %45, t45, %129, %45; fma.rn.f32 %46, t46, %129, %46; fma.rn.f32 %47, t47, %129, %47;\n\t"
      "fma.rn.f32 %48, t48, %129, %48; fma.rn.f32 %49, t49, %129, %49; fma.rn.f32 %50, t50, %129, %50; fma.rn.f32 %51, t51, %129, %51;\n\t"
      "fma.rn.f32 %52, t52, %129, %52; fma.rn.f32 %53, t53, %129, %53; fma.rn.f32 %54, t54, %129, %54; fma.rn.f32 %55, t55, %129, %55;\n\t"
      "fma.rn.f32 %56, t56, %129, %56; fma.rn.f32 %57, t57, %129, %57; fma.rn.f32 %58, t58, %129, %58; fma.rn.f32 %59, t59, %129, %59;\n\t"
      "fma.rn.f32 %60, t60, %129, %60; fma.rn.f32 %61, t61, %129, %61; fma.rn.f32 %62, t62, %129, %62; fma.rn.f32 %63, t63, %129, %63;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%128+96];\n\t"
      "fma.rn.f32 %64, t0, %129, %64; fma.rn.f32 %65, t1, %129, %65; fma.rn.f32 %66, t2, %129, %66; fma.rn.f32 %67, t3, %129, %67;\n\t"
      "fma.rn.f32 %68, t4, %129, %68; fma.rn.f32 %69, t5, %129, %69; fma.rn.f32 %70, t6, %129, %70; fma.rn.f32 %71, t7, %129, %71;\n\t"
      "fma.rn.f32 %72, t8, %129, %72; fma.rn.f32 %73, t9, %129, %73; fma.rn.f32 %74, t10, %129, %74; fma.rn.f32 %75, t11, %129, %75;\n\t"
      "fma.rn.f32 %76, t12, %129, %76; fma.rn.f32 %77, t13, %129, %77; fma.rn.f32 %78, t14, %129, %78; fma.rn.f32 %79, t15, %129, %79;\n\t"
      "fma.rn.f32 %80, t16, %129, %80; fma.rn.f32 %81, t17, %129, %81; fma.rn.f32 %82, t18, %129, %82; fma.rn.f32 %83, t19, %129, %83;\n\t"
      "fma.rn.f32 %84, t20, %129, %84; fma.rn.f32 %85, t21, %129, %85; fma.rn.f32 %86, t22, %129, %86; fma.rn.f32 %87, t23, %129, %87;\n\t"
      "fma.rn.f32 %88, t24, %129, %88; fma.rn.f32 %89, t25, %129, %89; fma.rn.f32 %90, t26, %129, %90; fma.rn.f32 %91, t27, %129, %91;\n\t"
      "fma.rn.f32 %92, t28, %129, %92; fma.rn.f32 %93, t29, %129, %93; fma.rn.f32 %94, t30, %129, %94; fma.rn.f32 %95, t31, %129, %95;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "fma.rn.f32 %96, t32, %129, %96; fma.rn.f32 %97, t33, %129, %97; fma.rn.f32 %98, t34, %129, %98; fma.rn.f32 %99, t35, %129, %99;\n\t"
      "fma.rn.f32 %100, t36, %129, %100; fma.rn.f32 %101, t37, %129, %101; fma.rn.f32 %102, t38, %129, %102; fma.rn.f32 %103, t39, %129, %103;\n\t"
      "fma.rn.f32 %104, t40, %129, %104; fma.rn.f32 %105, t41, %129, %105; fma.rn.f32 %106, t42, %129, %106; fma.rn.f32 %107, t43, %129, %107;\n\t"
      "fma.rn.f32 %108, t44, %129, %108; fma.rn.f32 %109, t45, %129, %109; fma.rn.f32 %110, t46, %129, %110; fma.rn.f32 %111, t47, %129, %111;\n\t"
      "fma.rn.f32 %112, t48, %129, %112; fma.rn.f32 %113, t49, %129, %113; fma.rn.f32 %114, t50, %129, %114; fma.rn.f32 %115, t51, %129, %115;\n\t"
      "fma.rn.f32 %116, t52, %129, %116; fma.rn.f32 %117, t53, %129, %117; fma.rn.f32 %118, t54, %129, %118; fma.rn.f32 %119, t55, %129, %119;\n\t"
      "fma.rn.f32 %120, t56, %129, %120; fma.rn.f32 %121, t57, %129, %121; fma.rn.f32 %122, t58, %129, %122; fma.rn.f32 %123, t59, %129, %123;\n\t"
      "fma.rn.f32 %124, t60, %129, %124; fma.rn.f32 %125, t61, %129, %125; fma.rn.f32 %126, t62, %129, %126; fma.rn.f32 %127, t63, %129, %127;\n\t"
      "}"
      : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]), "+f"(acc[7]),
        "+f"(acc[8]), "+f"(acc[9]), "+f"(acc[10]), "+f"(acc[11]), "+f"(acc[12]), "+f"(acc[13]), "+f"(acc[14]), "+f"(acc[15]),
        "+f"(acc[16]), "+f"(acc[17]), "+f"(acc[18]), "+f"(acc[19]), "+f"(acc[20]), "+f"(acc[21]), "+f"(acc[22]), "+f"(acc[23]),
        "+f"(acc[24]), "+f"(acc[25]), "+f"(acc[26]), "+f"(acc[27]), "+f"(acc[28]), "+f"(acc[29]), "+f"(acc[30]), "+f"(acc[31]),
        "+f"(acc[32]), "+f"(acc[33]), "+f"(acc[34]), "+f"(acc[35]), "+f"(acc[36]), "+f"(acc[37]), "+f"(acc[38]), "+f"(acc[39]),
        "+f"(acc[40]), "+f"(acc[41]), "+f"(acc[42]), "+f"(acc[43]), "+f"(acc[44]), "+f"(acc[45]), "+f"(acc[46]), "+f"(acc[47]),
        "+f"(acc[48]), "+f"(acc[49]), "+f"(acc[50]), "+f"(acc[51]), "+f"(acc[52]), "+f"(acc[53]), "+f"(acc[54]), "+f"(acc[55]),
        "+f"(acc[56]), "+f"(acc[57]), "+f"(acc[58]), "+f"(acc[59]), "+f"(acc[60]), "+f"(acc[61]), "+f"(acc[62]), "+f"(acc[63]),
        "+f"(acc[64]), "+f"(acc[65]), "+f"(acc[66]), "+f"(acc[67]), "+f"(acc[68]), "+f"(acc[69]), "+f"(acc[70]), "+f"(acc[71]),
        "+f"(acc[72]), "+f"(acc[73]), "+f"(acc[74]), "+f"(acc[75]), "+f"(acc[76]), "+f"(acc[77]), "+f"(acc[78]), "+f"(acc[79]),
        "+f"(acc[80]), "+f"(acc[81]), "+f"(acc[82]), "+f"(acc[83]), "+f"(acc[84]), "+f"(acc[85]), "+f"(acc[86]), "+f"(acc[87]),
        "+f"(acc[88]), "+f"(acc[89]), "+f"(acc[90]), "+f"(acc[91]), "+f"(acc[92]), "+f"(acc[93]), "+f"(acc[94]), "+f"(acc[95]),
        "+f"(acc[96]), "+f"(acc[97]), "+f"(acc[98]), "+f"(acc[99]), "+f"(acc[100]), "+f"(acc[101]), "+f"(acc[102]), "+f"(acc[103]),
        "+f"(acc[104]), "+f"(acc[105]), "+f"(acc[106]), "+f"(acc[107]), "+f"(acc[108]), "+f"(acc[109]), "+f"(acc[110]), "+f"(acc[111]),
        "+f"(acc[112]), "+f"(acc[113]), "+f"(acc[114]), "+f"(acc[115]), "+f"(acc[116]), "+f"(acc[117]), "+f"(acc[118]), "+f"(acc[119]),
        "+f"(acc[120]), "+f"(acc[121]), "+f"(acc[122]), "+f"(acc[123]), "+f"(acc[124]), "+f"(acc[125]), "+f"(acc[126]), "+f"(acc[127])
      : "r"(taddr), "f"(sc)
      : "memory");
}

MOE_DEV void tmem_fold128x2(uint32_t taddr, float sc, unsigned long long (&acc)[64]) {
  asm volatile(
      "{\n\t.reg .b32 t<64>;\n\t.reg .b64 s2, pt;\n\tmov.b64 s2, {%65, %65};\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%64+0];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%64+32];\n\t"
      "mov.b64 pt, {t0, t1}; fma.rn.f32x2 %0, pt, s2, %0; mov.b64 pt, {t2, t3}; fma.rn.f32x2 %1, pt, s2, %1; mov.b64 pt, {t4, t5}; fma.rn.f32x2 %2, pt, s2, %2; mov.b64 pt, {t6, t7}; fma.rn.f32x2 %3, pt, s2, %3;\n\t"
      "mov.b64 pt, {t8, t9}; fma.rn.f32x2 %4, pt, s2, %4; mov.b64 pt, {t10, t11}; fma.rn.f32x2 %5, pt, s2, %5; mov.b64 pt, {t12, t13}; fma.rn.f32x2 %6, pt, s2, %6; mov.b64 pt, {t14, t15}; fma.rn.f32x2 %7, pt, s2, %7;\n\t"
      "mov.b64 pt, {t16, t17}; fma.rn.f32x2 %8, pt, s2, %8; mov.b64 pt, {t18, t19}; fma.rn.f32x2 %9, pt, s2, %9; mov.b64 pt, {t20, t21}; fma.rn.f32x2 %10, pt, s2, %10; mov.b64 pt, {t22, t23}; fma.rn.f32x2 %11, pt, s2, %11;\n\t"
      "mov.b64 pt, {t24, t25}; fma.rn.f32x2 %12, pt, s2, %12; mov.b64 pt, {t26, t27}; fma.rn.f32x2 %13, pt, s2, %13; mov.b64 pt, {t28, t29}; fma.rn.f32x2 %14, pt, s2, %14; mov.b64 pt, {t30, t31}; fma.rn.f32x2 %15, pt, s2, %15;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%64+64];\n\t"
      "mov.b64 pt, {t32, t33}; fma.rn.f32x2 %16, pt, s2, %16; mov.b64 pt, {t34, t35}; fma.rn.f32x2 %17, pt, s2, %17; mov.b64 pt, {t36, t37}; fma.rn.f32x2 %18, pt, s2, %18; mov.b64 pt, {t38, t39}; fma.rn.f32x2 %19, pt, s2, %19;\n\t"
      "mov.b64 pt, {t40, t41}; fma.rn.f32x2 %20, pt, s2, %20; mov.b64 pt, {t42, t43}; fma.rn.f32x2 %21, pt, s2, %21; mov.b64 pt, {t44, t45}; fma.rn.f32x2 %22, pt, s2, %22; mov.b64 pt, {t46, t47}; fma.rn.f32x2 %23, pt, s2, %23;\n\t"
      "mov.b64 pt, {t48, t49}; fma.rn.f32x2 %24, pt, s2, %24; mov.b64 pt, {t50, t51}; fma.rn.f32x2 %25, pt, s2, %25; mov.b64 pt, {t52, t53}; fma.rn.f32x2 %26, pt, s2, %26; mov.b64 pt, {t54, t55}; fma.rn.f32x2 %27, pt, s2, %27;\n\t"
      "mov.b64 pt, {t56, t57}; fma.rn.f32x2 %28, pt, s2, %28; mov.b64 pt, {t58, t59}; fma.rn.f32x2 %29, pt, s2, %29; mov.b64 pt, {t60, t61}; fma.rn.f32x2 %30, pt, s2, %30; mov.b64 pt, {t62, t63}; fma.rn.f32x2 %31, pt, s2, %31;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t32, t33, t34, t35, t36, t37, t38, t39, t40, t41, t42, t43, t44, t45, t46, t47, t48, t49, t50, t51, t52, t53, t54, t55, t56, t57, t58, t59, t60, t61, t62, t63}, [%64+96];\n\t"
      "mov.b64 pt, {t0, t1}; fma.rn.f32x2 %32, pt, s2, %32; mov.b64 pt, {t2, t3}; fma.rn.f32x2 %33, pt, s2, %33; mov.b64 pt, {t4, t5}; fma.rn.f32x2 %34, pt, s2, %34; mov.b64 pt, {t6, t7}; fma.rn.f32x2 %35, pt, s2, %35;\n\t"
      "mov.b64 pt, {t8, t9}; fma.rn.f32x2 %36, pt, s2, %36; mov.b64 pt, {t10, t11}; fma.rn.f32x2 %37, pt, s2, %37; mov.b64 pt, {t12, t13}; fma.rn.f32x2 %38, pt, s2, %38; mov.b64 pt, {t14, t15}; fma.rn.f32x2 %39, pt, s2, %39;\n\t"
      "mov.b64 pt, {t16, t17}; fma.rn.f32x2 %40, pt, s2, %40; mov.b64 pt, {t18, t19}; fma.rn.f32x2 %41, pt, s2, %41; mov.b64 pt, {t20, t21}; fma.rn.f32x2 %42, pt, s2, %42; mov.b64 pt, {t22, t23}; fma.rn.f32x2 %43, pt, s2, %43;\n\t"
      "mov.b64 pt, {t24, t25}; fma.rn.f32x2 %44, pt, s2, %44; mov.b64 pt, {t26, t27}; fma.rn.f32x2 %45, pt, s2, %45; mov.b64 pt, {t28, t29}; fma.rn.f32x2 %46, pt, s2, %46; mov.b64 pt, {t30, t31}; fma.rn.f32x2 %47, pt, s2, %47;\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 pt, {t32, t33}; fma.rn.f32x2 %48, pt, s2, %48; mov.b64 pt, {t34, t35}; fma.rn.f32x2 %49, pt, s2, %49; mov.b64 pt, {t36, t37}; fma.rn.f32x2 %50, pt, s2, %50; mov.b64 pt, {t38, t39}; fma.rn.f32x2 %51, pt, s2, %51;\n\t"
      "mov.b64 pt, {t40, t41}; fma.rn.f32x2 %52, pt, s2, %52; mov.b64 pt, {t42, t43}; fma.rn.f32x2 %53, pt, s2, %53; mov.b64 pt, {t44, t45}; fma.rn.f32x2 %54, pt, s2, %54; mov.b64 pt, {t46, t47}; fma.rn.f32x2 %55, pt, s2, %55;\n\t"
      "mov.b64 pt, {t48, t49}; fma.rn.f32x2 %56, pt, s2, %56; mov.b64 pt, {t50, t51}; fma.rn.f32x2 %57, pt, s2, %57; mov.b64 pt, {t52, t53}; fma.rn.f32x2 %58, pt, s2, %58; mov.b64 pt, {t54, t55}; fma.rn.f32x2 %59, pt, s2, %59;\n\t"
      "mov.b64 pt, {t56, t57}; fma.rn.f32x2 %60, pt, s2, %60; mov.b64 pt, {t58, t59}; fma.rn.f32x2 %61, pt, s2, %61; mov.b64 pt, {t60, t61}; fma.rn.f32x2 %62, pt, s2, %62; mov.b64 pt, {t62, t63}; fma.rn.f32x2 %63, pt, s2, %63;\n\t"
      "}"
      : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7]),
        "+l"(acc[8]), "+l"(acc[9]), "+l"(acc[10]), "+l"(acc[11]), "+l"(acc[12]), "+l"(acc[13]), "+l"(acc[14]), "+l"(acc[15]),
        "+l"(acc[16]), "+l"(acc[17]), "+l"(acc[18]), "+l"(acc[19]), "+l"(acc[20]), "+l"(acc[21]), "+l"(acc[22]), "+l"(acc[23]),
        "+l"(acc[24]), "+l"(acc[25]), "+l"(acc[26]), "+l"(acc[27]), "+l"(acc[28]), "+l"(acc[29]), "+l"(acc[30]), "+l"(acc[31]),
        "+l"(acc[32]), "+l"(acc[33]), "+l"(acc[34]), "+l"(acc[35]), "+l"(acc[36]), "+l"(acc[37]), "+l"(acc[38]), "+l"(acc[39]),
        "+l"(acc[40]), "+l"(acc[41]), "+l"(acc[42]), "+l"(acc[43]), "+l"(acc[44]), "+l"(acc[45]), "+l"(acc[46]), "+l"(acc[47]),
        "+l"(acc[48]), "+l"(acc[49]), "+l"(acc[50]), "+l"(acc[51]), "+l"(acc[52]), "+l"(acc[53]), "+l"(acc[54]), "+l"(acc[55]),
        "+l"(acc[56]), "+l"(acc[57]), "+l"(acc[58]), "+l"(acc[59]), "+l"(acc[60]), "+l"(acc[61]), "+l"(acc[62]), "+l"(acc[63])
      : "r"(taddr), "f"(sc)
      : "memory");
}

// tmem_fold32x2: the transposed form.  acc[i] (i < 16, packed pairs as in
// tmem_fold128x2) += 32 consecutive fp32 TMEM columns of this thread's lane
// times a per-column scale, c[i] holding the scales of columns 2i and 2i+1.
MOE_DEV void tmem_fold32x2(uint32_t taddr, const unsigned long long (&c)[16], unsigned long long (&acc)[64]) {
  asm volatile(
      "{\n\t.reg .b32 t<32>;\n\t.reg .b64 pt;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 pt, {t0, t1}; fma.rn.f32x2 %0, pt, %17, %0; mov.b64 pt, {t2, t3}; fma.rn.f32x2 %1, pt, %18, %1; mov.b64 pt, {t4, t5}; fma.rn.f32x2 %2, pt, %19, %2; mov.b64 pt, {t6, t7}; fma.rn.f32x2 %3, pt, %20, %3;\n\t"
      "mov.b64 pt, {t8, t9}; fma.rn.f32x2 %4, pt, %21, %4; mov.b64 pt, {t10, t11}; fma.rn.f32x2 %5, pt, %22, %5; mov.b64 pt, {t12, t13}; fma.rn.f32x2 %6, pt, %23, %6; mov.b64 pt, {t14, t15}; fma.rn.f32x2 %7, pt, %24, %7;\n\t"
      "mov.b64 pt, {t16, t17}; fma.rn.f32x2 %8, pt, %25, %8; mov.b64 pt, {t18, t19}; fma.rn.f32x2 %9, pt, %26, %9; mov.b64 pt, {t20, t21}; fma.rn.f32x2 %10, pt, %27, %10; mov.b64 pt, {t22, t23}; fma.rn.f32x2 %11, pt, %28, %11;\n\t"
      "mov.b64 pt, {t24, t25}; fma.rn.f32x2 %12, pt, %29, %12; mov.b64 pt, {t26, t27}; fma.rn.f32x2 %13, pt, %30, %13; mov.b64 pt, {t28, t29}; fma.rn.f32x2 %14, pt, %31, %14; mov.b64 pt, {t30, t31}; fma.rn.f32x2 %15, pt, %32, %15;\n\t"
      "}"
      : "+l"(acc[0]), "+l"(acc[1]), "+l"(acc[2]), "+l"(acc[3]), "+l"(acc[4]), "+l"(acc[5]), "+l"(acc[6]), "+l"(acc[7]), "+l"(acc[8]), "+l"(acc[9]), "+l"(acc[10]), "+l"(acc[11]), "+l"(acc[12]), "+l"(acc[13]), "+l"(acc[14]), "+l"(acc[15])
      : "r"(taddr), "l"(c[0]), "l"(c[1]), "l"(c[2]), "l"(c[3]), "l"(c[4]), "l"(c[5]), "l"(c[6]), "l"(c[7]), "l"(c[8]), "l"(c[9]), "l"(c[10]), "l"(c[11]), "l"(c[12]), "l"(c[13]), "l"(c[14]), "l"(c[15])
      : "memory");
}

// tmem_fold32: tmem_fold32x2 with scalar accumulators (acc[0..31], column t
// in acc[t]) and fma.rn.f32; the same sums bit for bit.
MOE_DEV void tmem_fold32(uint32_t taddr, const unsigned long long (&c)[16], float (&acc)[128]) {
  asm volatile(
      "{\n\t.reg .b32 t<32>;\n\t.reg .b32 cl, ch;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 {cl, ch}, %33; fma.rn.f32 %0, t0, cl, %0; fma.rn.f32 %1, t1, ch, %1; mov.b64 {cl, ch}, %34; fma.rn.f32 %2, t2, cl, %2; fma.rn.f32 %3, t3, ch, %3; mov.b64 {cl, ch}, %35; fma.rn.f32 %4, t4, cl, %4; fma.rn.f32 %5, t5, ch, %5; mov.b64 {cl, ch}, %36; fma.rn.f32 %6, t6, cl, %6; fma.rn.f32 %7, t7, ch, %7;\n\t"
      "mov.b64 {cl, ch}, %37; fma.rn.f32 %8, t8, cl, %8; fma.rn.f32 %9, t9, ch, %9; mov.b64 {cl, ch}, %38; fma.rn.f32 %10, t10, cl, %10; fma.rn.f32 %11, t11, ch, %11; mov.b64 {cl, ch}, %39; fma.rn.f32 %12, t12, cl, %12; fma.rn.f32 %13, t13, ch, %13; mov.b64 {cl, ch}, %40; fma.rn.f32 %14, t14, cl, %14; fma.rn.f32 %15, t15, ch, %15;\n\t"
      "mov.b64 {cl, ch}, %41; fma.rn.f32 %16, t16, cl, %16; fma.rn.f32 %17, t17, ch, %17; mov.b64 {cl, ch}, %42; fma.rn.f32 %18, t18, cl, %18; fma.rn.f32 %19, t19, ch, %19; mov.b64 {cl, ch}, %43; fma.rn.f32 %20, t20, cl, %20; fma.rn.f32 %21, t21, ch, %21; mov.b64 {cl, ch}, %44; fma.rn.f32 %22, t22, cl, %22; fma.rn.f32 %23, t23, ch, %23;\n\t"
      "mov.b64 {cl, ch}, %45; fma.rn.f32 %24, t24, cl, %24; fma.rn.f32 %25, t25, ch, %25; mov.b64 {cl, ch}, %46; fma.rn.f32 %26, t26, cl, %26; fma.rn.f32 %27, t27, ch, %27; mov.b64 {cl, ch}, %47; fma.rn.f32 %28, t28, cl, %28; fma.rn.f32 %29, t29, ch, %29; mov.b64 {cl, ch}, %48; fma.rn.f32 %30, t30, cl, %30; fma.rn.f32 %31, t31, ch, %31;\n\t"
      "}"
      : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]), "+f"(acc[7]), "+f"(acc[8]), "+f"(acc[9]), "+f"(acc[10]), "+f"(acc[11]), "+f"(acc[12]), "+f"(acc[13]), "+f"(acc[14]), "+f"(acc[15]), "+f"(acc[16]), "+f"(acc[17]), "+f"(acc[18]), "+f"(acc[19]), "+f"(acc[20]), "+f"(acc[21]), "+f"(acc[22]), "+f"(acc[23]), "+f"(acc[24]), "+f"(acc[25]), "+f"(acc[26]), "+f"(acc[27]), "+f"(acc[28]), "+f"(acc[29]), "+f"(acc[30]), "+f"(acc[31])
      : "r"(taddr), "l"(c[0]), "l"(c[1]), "l"(c[2]), "l"(c[3]), "l"(c[4]), "l"(c[5]), "l"(c[6]), "l"(c[7]), "l"(c[8]), "l"(c[9]), "l"(c[10]), "l"(c[11]), "l"(c[12]), "l"(c[13]), "l"(c[14]), "l"(c[15])
      : "memory");
}

}  // namespace moe
