"""Float64 CPU oracle for the hybrid sparse MQA attention step.

Test infrastructure only: tests, the smoke check and the benchmark's CPU
baseline leg use it; the library never does.
"""
