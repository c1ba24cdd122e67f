#!/bin/bash
cd $GRAFT_REPO_ROOT
python -c "import __graft_entry__ as g; g.build()" > gpurun_out/build.log 2>&1 || { tail -30 gpurun_out/build.log; exit 1; }
cd _work
timeout 300 python checkvar.py ../tree_verification_attention_gb300/libtva.so > ../gpurun_out/check.log 2>&1; rc0=$?
tail -2 ../gpurun_out/check.log
[ $rc0 -eq 0 ] || exit $rc0
python mkvar.py timeline > ../gpurun_out/mkvar.log 2>&1 || { tail -20 ../gpurun_out/mkvar.log; exit 1; }
timeout 300 python tl.py var/timeline/libtva.so 3 2>&1 | tail -12; rc=${PIPESTATUS[0]}
for i in 1 2; do timeout 300 python timevar.py ../tree_verification_attention_gb300/libtva.so 3; done
exit $rc
